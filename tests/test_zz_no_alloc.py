"""The allocation-free decode attention entry point (GPU).

llama_op_attention_decode_noalloc serves callers that cannot allocate device
memory when they run attention: it keeps its split-KV partials in the
library's own fixed-size device array.  This file is collected last so that a
run stopping at the first failure has already run every other test; it loads
the library itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import synth
from _helpers import assert_parity, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu


def _case(B, start_pos, H, G, D, tag):
    L = start_pos + 3
    q = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/q{tag}", (B, 1, H, D)))
    kc = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/k{tag}", (B, G, L, D)))
    vc = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/v{tag}", (B, G, L, D)))
    return to_dev(q), to_dev(kc), to_dev(vc), L


def _existing(lb, q, kd, vd, L, B, start_pos, H, G, D):
    """Output of the existing entry point, with a caller-provided workspace."""
    t = torch()
    o = t.empty_like(q)
    n = lb.llama_op_attention_workspace_bytes(lb.LLAMA_BF16, B, 1, start_pos, H, D)
    ws = t.empty(max(n, 16), dtype=t.uint8, device="cuda")
    lb.check(lb.llama_op_attention(lb.LLAMA_BF16, q, lb.make_kv_cache(kd, vd, B, L), o, B, 1, start_pos, H, G, D,
                                   ws, n))
    return o


def test_noalloc_decode_matches_existing_entry_point_on_consecutive_calls():
    import decoder_block_gb300 as lb
    lb.load()
    t = torch()
    # two calls in a row with different shapes: the second must not see the
    # first call's partials (the array keeps the last call's contents)
    cases = [(8, 1500, 32, 8, 128, "a"), (3, 700, 9, 3, 64, "b"), (8, 1500, 32, 8, 128, "a")]
    for B, sp, H, G, D, tag in cases:
        q, kd, vd, L = _case(B, sp, H, G, D, tag)
        ref = _existing(lb, q, kd, vd, L, B, sp, H, G, D)
        o = t.full_like(q, float("nan"))
        lb.check(lb.llama_op_attention_decode_noalloc(q, lb.make_kv_cache(kd, vd, B, L), o, B, sp, H, G, D),
                 "llama_op_attention_decode_noalloc")
        t.cuda.synchronize()
        got, want = to_f64(o), to_f64(ref)
        assert_parity(got, want, "bf16", f"noalloc vs existing entry point B={B} start_pos={sp} H={H} D={D}")
        assert np.all(np.isfinite(got))


def test_noalloc_rejects_requests_beyond_its_array():
    import decoder_block_gb300 as lb
    lb.load()
    t = torch()
    q = t.zeros((64, 32, 128), dtype=t.bfloat16, device="cuda")
    kc = t.zeros((64, 8, 16, 128), dtype=t.bfloat16, device="cuda")
    kv = lb.make_kv_cache(kc, kc, 64, 20000)  # claims 20000 positions: partials need > 32 MiB
    need = 64 * 32 * ((16000 + 255) // 256) * 130 * 4
    assert need > lb.LLAMA_NOALLOC_SCRATCH_BYTES
    assert lb.llama_op_attention_decode_noalloc(q, kv, q, 64, 15999, 32, 8, 128) == lb.LLAMA_ERR_RANGE
