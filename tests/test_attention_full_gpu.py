"""Element-wise parity of the d_head-128 causal GQA prefill attention at the
8B prefill sequence lengths ([EVT] §05 GQA; [L3B] How it works: the causal
mask over the cache), through llama_op_attention, against the fp64 oracle.

B = 1, S = 8192 and B = 4, S = 2048 with H = 32, G = 8: every query row of
every head is compared (the persistent kernel's schedule at S = 8192 gives
each CTA about 219 key tiles from several query blocks, all of them covered
here).  The oracle runs head by head on a few host threads (each S x S fp64
score matrix is 0.5 GB at S = 8192).
"""
import concurrent.futures

import numpy as np
import pytest

import oracle
import synth
from _helpers import assert_parity, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


@pytest.mark.parametrize("B,S", [(1, 8192), (4, 2048)])
def test_prefill_attention_d128_full_length(lb, B, S):
    t = torch()
    H, G, D = 32, 8, 128
    r = H // G
    q = synth.f32_to_bf16_bits(synth.normal(0, f"full/q{B}", (B, S, H, D)))
    kc = synth.f32_to_bf16_bits(synth.normal(0, f"full/k{B}", (B, G, S, D)))
    vc = synth.f32_to_bf16_bits(synth.normal(0, f"full/v{B}", (B, G, S, D)))
    qd, kd, vd = to_dev(q), to_dev(kc), to_dev(vc)
    o = t.full_like(qd, float("nan"))
    assert lb.llama_op_attention_workspace_bytes(lb.LLAMA_BF16, B, S, 0, H, D) == 0
    lb.check(lb.llama_op_attention(lb.LLAMA_BF16, qd, lb.make_kv_cache(kd, vd, B, S), o, B, S, 0, H, G, D,
                                   t.empty(16, dtype=t.uint8, device="cuda"), 0))
    t.cuda.synchronize()
    got = to_f64(o)
    q64, k64, v64 = synth.as_f64(q), synth.as_f64(kc), synth.as_f64(vc)

    def one(bh):
        b, h = bh
        g = h // r
        return bh, oracle.gqa_attention(q64[b:b + 1, :, h:h + 1], k64[b:b + 1, g:g + 1], v64[b:b + 1, g:g + 1],
                                        0)[0, :, 0]

    ref = np.empty((B, S, H, D))
    with concurrent.futures.ThreadPoolExecutor(max_workers=4) as ex:
        for (b, h), o_bh in ex.map(one, [(b, h) for b in range(B) for h in range(H)]):
            ref[b, :, h] = o_bh
    assert_parity(got, ref, "bf16", f"attention B={B} S={S} (all rows)")
    for b in range(B):
        for h in range(H):
            assert_parity(got[b, :, h], ref[b, :, h], "bf16", f"attention B={B} S={S} b={b} h={h}")
