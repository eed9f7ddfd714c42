"""The fused decode-step kernel (LLAMA_DECODE_FUSED) against the fp64 oracle (GPU).

"Full Llama 3 transformer block", How it works: a decode step feeds one new
token per sequence through the block, attending to the cached keys
0 .. start_pos.  With the fused mode set, an S = 1 forward of a dense bf16
block with d_head = 128 runs as one cooperative kernel; these tests check
- y and the written cache entry against the oracle (bf16 parity bars), every
  other cache position unchanged, across batch sizes and cache lengths that
  give one or several 512-key chunks and a ragged last chunk;
- that the fused and the multi-kernel path agree closely (same device code,
  same tile plans; only the order of fp32 reductions may differ);
- the full-size Llama-3-8B decode step (B = 64 at position 4095);
- the mode switch: unknown modes are rejected, prefill and ineligible blocks
  keep running as separate kernels, and the fused forward is one launch.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import (GpuBlock, assert_branch_parity, assert_parity, f64_weights, parity_errors, to_dev, to_f64,
                      torch)

pytestmark = pytest.mark.gpu

# d_head 128 (the fused kernel's), GQA groups of 4 and 2, reduced widths
SHAPES = {
    "d1024_gqa4": dict(d_model=1024, n_heads=8, n_kv_heads=2, d_ff=2816, norm_eps=1e-5, rope_theta=5e5,
                       dtype="bf16", max_seq_len=2048),
    "d2048_gqa2": dict(d_model=2048, n_heads=16, n_kv_heads=8, d_ff=5632, norm_eps=1e-5, rope_theta=5e5,
                       dtype="bf16", max_seq_len=2048),
}


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


def _decode(lb, shape, w, x, kc, vc, B, start_pos, mode):
    t = torch()
    with GpuBlock(shape, w, B, max_seq_len=kc.shape[2]) as blk:
        lb.check(lb.llama_block_set_decode_mode(blk.h, mode), "llama_block_set_decode_mode")
        xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
        yd = t.empty_like(xd)
        n0 = lb.llama_kernel_launch_count()
        lb.check(blk.forward(xd, yd, B, 1, start_pos, kd, vd), "llama_block_forward")
        launches = lb.llama_kernel_launch_count() - n0
        t.cuda.synchronize()
        lb.check(lb.llama_block_device_status(blk.h), "device status")
        return to_f64(yd), to_f64(kd), to_f64(vd), launches


@pytest.mark.parametrize("name,B,start_pos,L", [
    ("d1024_gqa4", 1, 0, 64),        # first token: one key
    ("d1024_gqa4", 3, 37, 64),       # one chunk, ragged tile
    ("d1024_gqa4", 5, 511, 600),     # exactly one full chunk
    ("d1024_gqa4", 2, 1300, 1400),   # three chunks, ragged last one
    ("d2048_gqa2", 64, 700, 800),    # decode batch, two chunks
    ("d2048_gqa2", 130, 90, 128),    # more rows than one 128-row tile
])
def test_fused_decode_matches_oracle(lb, name, B, start_pos, L):
    s = SHAPES[name]
    w = synth.block_weights(s)
    x = synth.block_activations(s, tag=f"fused_{B}_{start_pos}", B=B, S=1)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=L, fill_upto=start_pos)
    y, kg, vg, launches = _decode(lb, s, w, x, kc, vc, B, start_pos, lb.LLAMA_DECODE_FUSED)
    assert launches == 1
    yr, kr, vr = oracle.block_forward(s, f64_weights(w), synth.as_f64(x), start_pos, synth.as_f64(kc),
                                      synth.as_f64(vc))
    assert_parity(y, yr, "bf16", "y")
    assert_branch_parity(y, yr, synth.as_f64(x), "y - x (both branch outputs)")
    sl = (slice(0, B), slice(None), slice(start_pos, start_pos + 1))
    assert_parity(kg[sl], kr[sl], "bf16", "K cache entry")
    assert_parity(vg[sl], vr[sl], "bf16", "V cache entry")
    untouched = np.ones(kg.shape, dtype=bool)
    untouched[sl] = False
    np.testing.assert_array_equal(kg[untouched], synth.as_f64(kc)[untouched])
    np.testing.assert_array_equal(vg[untouched], synth.as_f64(vc)[untouched])


@pytest.mark.parametrize("layout", ["interleaved", "halves"])
def test_fused_equals_multi_kernel_path(lb, layout):
    s = dict(SHAPES["d1024_gqa4"], rope_layout=layout)
    B, sp, L = 16, 900, 1024
    w = synth.block_weights(s)
    x = synth.block_activations(s, tag="fused_vs_kernels", B=B, S=1)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=L, fill_upto=sp)
    yf, kf, vf, nf = _decode(lb, s, w, x, kc, vc, B, sp, lb.LLAMA_DECODE_FUSED)
    yk, kk, vk, nk = _decode(lb, s, w, x, kc, vc, B, sp, lb.LLAMA_DECODE_KERNELS)
    assert nf == 1 and nk == 7
    # K and V of the new token come from the same GEMM epilogue code and plan:
    # only the split-K reduction order differs (fp32), so at most one bf16 ulp
    fro, mx = parity_errors(kf, kk)
    assert fro <= 2e-3 and mx <= 1e-2, (fro, mx)
    fro, mx = parity_errors(yf - synth.as_f64(x), yk - synth.as_f64(x))
    assert fro <= 5e-3, fro
    yr, _, _ = oracle.block_forward(s, f64_weights(w), synth.as_f64(x), sp, synth.as_f64(kc), synth.as_f64(vc))
    assert_parity(yf, yr, "bf16", "y (fused)")


def test_fused_llama3_8b_decode_full_size(lb):
    s = synth.SHAPES["llama3_8b_decode_b64"]
    B, sp = s["B"], s["start_pos"]
    w = synth.block_weights(s)
    x = synth.block_activations(s)
    kc, vc = synth.kv_cache(s, fill_upto=sp)
    y, kg, vg, launches = _decode(lb, s, w, x, kc, vc, B, sp, lb.LLAMA_DECODE_FUSED)
    assert launches == 1
    rows = [(b, 0) for b in range(B)]
    yr, kr, vr = oracle.block_forward_rows(s, f64_weights(w), synth.as_f64(x), sp, synth.as_f64(kc),
                                           synth.as_f64(vc), rows)
    assert_parity(y[:, 0], yr, "bf16", "y")
    assert_branch_parity(y[:, 0], yr, synth.as_f64(x)[:, 0], "y - x")
    assert_parity(kg[:, :, sp:sp + 1], kr, "bf16", "K cache entry")
    assert_parity(vg[:, :, sp:sp + 1], vr, "bf16", "V cache entry")
    np.testing.assert_array_equal(kg[:, :, :sp], synth.as_f64(kc)[:, :, :sp])


def test_decode_mode_switch(lb):
    t = torch()
    s = SHAPES["d1024_gqa4"]
    w = synth.block_weights(s)
    with GpuBlock(s, w, 64, max_seq_len=128) as blk:
        assert lb.llama_block_set_decode_mode(blk.h, 7) == lb.LLAMA_ERR_INVALID_ARG
        assert lb.llama_block_set_decode_mode(None, lb.LLAMA_DECODE_FUSED) == lb.LLAMA_ERR_INVALID_ARG
        lb.check(lb.llama_block_set_decode_mode(blk.h, lb.LLAMA_DECODE_FUSED))
        # a prefill chunk (S > 1) still runs as separate kernels
        x = synth.block_activations(s, tag="mode_prefill", B=2, S=20)
        kc, vc = synth.kv_cache(s, max_batch=2, max_seq_len=128)
        xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
        yd = t.empty_like(xd)
        n0 = lb.llama_kernel_launch_count()
        lb.check(blk.forward(xd, yd, 2, 20, 0, kd, vd))
        assert lb.llama_kernel_launch_count() - n0 == 6
        t.cuda.synchronize()
        yr, _, _ = oracle.block_forward(s, f64_weights(w), synth.as_f64(x), 0, synth.as_f64(kc), synth.as_f64(vc))
        assert_parity(to_f64(yd), yr, "bf16", "prefill y with the fused decode mode set")
    # d_head 64 (SmolLM2-shaped): the fused kernel does not apply; decode keeps its kernels
    s2 = dict(synth.SHAPES["smollm2_135m"], max_seq_len=64)
    w2 = synth.block_weights(s2)
    x2 = synth.block_activations(s2, tag="mode_d64", B=4, S=1)
    kc2, vc2 = synth.kv_cache(s2, max_batch=4, max_seq_len=64, fill_upto=30)
    y2, _, _, n2 = _decode(lb, s2, w2, x2, kc2, vc2, 4, 30, lb.LLAMA_DECODE_FUSED)
    assert n2 > 1
    yr2, _, _ = oracle.block_forward(s2, f64_weights(w2), synth.as_f64(x2), 30, synth.as_f64(kc2),
                                     synth.as_f64(vc2))
    assert_parity(y2, yr2, "bf16", "d_head 64 decode with the fused mode set")


def test_fused_decode_chain_and_y_aliasing_x(lb):
    """Several consecutive steps on one handle (the barrier words are re-armed
    by every launch), y written over x."""
    t = torch()
    s = SHAPES["d1024_gqa4"]
    B, L, sp0 = 4, 96, 60
    w = synth.block_weights(s)
    wf = f64_weights(w)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=L, fill_upto=sp0)
    kr, vr = synth.as_f64(kc), synth.as_f64(vc)
    with GpuBlock(s, w, B, max_seq_len=L) as blk:
        lb.check(lb.llama_block_set_decode_mode(blk.h, lb.LLAMA_DECODE_FUSED))
        kd, vd = to_dev(kc), to_dev(vc)
        for step in range(4):
            x = synth.block_activations(s, tag=f"chain_{step}", B=B, S=1)
            xd = to_dev(x)
            lb.check(blk.forward(xd, xd, B, 1, sp0 + step, kd, vd))
            t.cuda.synchronize()
            yr, kr, vr = oracle.block_forward(s, wf, synth.as_f64(x), sp0 + step, kr, vr)
            assert_parity(to_f64(xd), yr, "bf16", f"step {step} y (aliasing x)")
        lb.check(lb.llama_block_device_status(blk.h))
        assert_parity(to_f64(kd)[:, :, sp0:sp0 + 4], kr[:, :, sp0:sp0 + 4], "bf16", "K cache after the chain")
