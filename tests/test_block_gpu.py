"""Whole-block parity of the C-ABI forward against the fp64 oracle (GPU).

Configurations: the tiny fp32 block, the SmolLM2-135M-shaped block, the
Llama-3-8B-shaped prefill (B=1 S=8192 and B=4 S=2048) and decode (B=64 at
start_pos 4095 over a pre-filled cache).  The full-size 8B cases compare every
written cache element and a sample of output rows that the oracle computes one
by one (first, last, tile edges and random rows).
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import GpuBlock, assert_branch_parity, assert_parity, f64_weights, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


def _run(shape, w, x, kc, vc, B, S, start_pos, max_tokens=None):
    t = torch()
    with GpuBlock(shape, w, max_tokens or B * S, max_seq_len=kc.shape[2]) as blk:
        xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
        yd = t.empty_like(xd)
        blk.lb.check(blk.forward(xd, yd, B, S, start_pos, kd, vd), "llama_block_forward")
        t.cuda.synchronize()
        blk.lb.check(blk.lb.llama_block_device_status(blk.h), "device status")
        return to_f64(yd), to_f64(kd), to_f64(vd)


def _check_full(shape, B, S, start_pos, L, fill_upto=0, tag="x"):
    w = synth.block_weights(shape)
    x = synth.block_activations(shape, tag=tag, B=B, S=S)
    kc, vc = synth.kv_cache(shape, max_batch=B, max_seq_len=L, fill_upto=fill_upto)
    y, kg, vg = _run(shape, w, x, kc, vc, B, S, start_pos)
    yr, kr, vr = oracle.block_forward(shape, f64_weights(w), synth.as_f64(x), start_pos, synth.as_f64(kc),
                                      synth.as_f64(vc))
    dt = shape["dtype"]
    assert_parity(y, yr, dt, "y")
    if dt == "bf16":
        assert_branch_parity(y, yr, synth.as_f64(x), "y - x (both branch outputs)")
    else:
        assert_parity(y - synth.as_f64(x), yr - synth.as_f64(x), dt, "y - x (both branch outputs)")
    sl = (slice(0, B), slice(None), slice(start_pos, start_pos + S))
    assert_parity(kg[sl], kr[sl], dt, "K cache slice")
    assert_parity(vg[sl], vr[sl], dt, "V cache slice")
    untouched = np.ones(kg.shape, dtype=bool)
    untouched[sl] = False
    np.testing.assert_array_equal(kg[untouched], synth.as_f64(kc)[untouched])
    np.testing.assert_array_equal(vg[untouched], synth.as_f64(vc)[untouched])


def test_tiny_f32_block():
    s = synth.SHAPES["tiny_f32"]
    _check_full(s, s["B"], s["S"], 0, s["max_seq_len"])


def test_smollm2_block_bf16():
    s = synth.SHAPES["smollm2_135m"]
    _check_full(s, s["B"], s["S"], 0, s["max_seq_len"])


@pytest.mark.parametrize("B,S,start_pos,L", [(2, 50, 0, 64), (3, 17, 30, 60), (1, 1, 0, 4), (4, 129, 0, 140)])
def test_ragged_and_offset_shapes_bf16(B, S, start_pos, L):
    s = dict(synth.SHAPES["smollm2_135m"], B=B, S=S, max_seq_len=L)
    _check_full(s, B, S, start_pos, L, fill_upto=start_pos, tag=f"xr{B}{S}")


LLAMA31_SCALING = dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)


@pytest.mark.parametrize("name,dtype", [("tiny_f32", "f32"), ("tiny_f32", "bf16"), ("smollm2_135m", "bf16")])
def test_halves_rope_layout_block(name, dtype):
    """Pairs (i, i + D/2): the CUDA-core path and the d_head-16 bf16 path rotate in the standalone kernel,
    the SmolLM2-shaped bf16 block in the QKV epilogue over reordered weight rows."""
    shape = dict(synth.SHAPES[name], dtype=dtype, rope_layout="halves")
    _check_full(shape, 2, 40, 0, 48, tag="halves")
    _check_full(shape, 3, 1, 30, 40, fill_upto=30, tag="halves_dec")


@pytest.mark.parametrize("layout", ["interleaved", "halves"])
def test_llama31_scaled_rope_past_the_original_context(layout):
    """Llama 3.1 frequency stretch at positions beyond the 8192 the unscaled model was trained at:
    a prefill chunk at 12000 and a decode step at 20000 over pre-filled caches."""
    shape = dict(synth.SHAPES["llama3_8b_prefill_b1s8192"], rope_layout=layout, rope_scaling=LLAMA31_SCALING,
                 max_seq_len=20004)
    _check_full(shape, 1, 40, 12000, 12040, fill_upto=12000, tag="scaled")
    _check_full(shape, 2, 1, 20000, 20004, fill_upto=20000, tag="scaled_dec")


def test_tiny_f32_decode_after_prefix():
    s = dict(synth.SHAPES["tiny_f32"], max_seq_len=24)
    _check_full(s, 2, 1, 9, 24, fill_upto=9, tag="xd")


def _sample_rows(B, S, n_random=12, seed=0):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (B - 1, S - 1), (0, min(S - 1, 127)), (0, min(S - 1, 128)), (B - 1, S // 2)}
    for _ in range(n_random):
        rows.add((int(rng.integers(B)), int(rng.integers(S))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["llama3_8b_prefill_b1s8192", "llama3_8b_prefill_b4s2048"])
def test_llama3_8b_prefill_full_size_sampled(name):
    s = synth.SHAPES[name]
    B, S = s["B"], s["S"]
    w = synth.block_weights(s)
    x = synth.block_activations(s)
    kc, vc = synth.kv_cache(s)
    y, kg, vg = _run(s, w, x, kc, vc, B, S, 0)
    rows = _sample_rows(B, S)
    yr, kr, vr = oracle.block_forward_rows(s, f64_weights(w), synth.as_f64(x), 0, synth.as_f64(kc),
                                           synth.as_f64(vc), rows)
    ys = np.stack([y[b, t] for b, t in rows])
    xs = np.stack([synth.as_f64(x)[b, t] for b, t in rows])
    assert_parity(ys, yr, "bf16", "y (sampled rows)")
    assert_branch_parity(ys, yr, xs, "y - x (sampled rows)")
    assert_parity(kg[:, :, :S], kr, "bf16", "K cache (all written positions)")
    assert_parity(vg[:, :, :S], vr, "bf16", "V cache (all written positions)")


def test_llama3_8b_ragged_prefill_on_cta_pairs():
    """B=2, S=2250 (4500 rows: the last 256-row pair tile has 148 live rows, 20 of them in its second
    CTA) at start_pos 100 over a filled cache prefix: all four GEMMs run on CTA pairs.  Sampled rows
    at both ends of that tile, every written K/V element, and the prefix bit for bit."""
    s = dict(synth.SHAPES["llama3_8b_prefill_b4s2048"], B=2, S=2250, max_seq_len=2400)
    B, S, sp = 2, 2250, 100
    w = synth.block_weights(s)
    x = synth.block_activations(s, tag="ragged_pairs", B=B, S=S)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=2400, fill_upto=sp)
    y, kg, vg = _run(s, w, x, kc, vc, B, S, sp)
    rows = sorted({(0, 0), (0, 2249), (1, 0), (1, 2101), (1, 2102), (1, 2229), (1, 2230), (1, 2249)} |
                  set(_sample_rows(B, S, n_random=6, seed=3)))
    yr, kr, vr = oracle.block_forward_rows(s, f64_weights(w), synth.as_f64(x), sp, synth.as_f64(kc),
                                           synth.as_f64(vc), rows)
    ys = np.stack([y[b, t] for b, t in rows])
    xs = np.stack([synth.as_f64(x)[b, t] for b, t in rows])
    assert_parity(ys, yr, "bf16", "y (sampled rows)")
    assert_branch_parity(ys, yr, xs, "y - x (sampled rows)")
    assert_parity(kg[:, :, sp:sp + S], kr, "bf16", "K cache (all written positions)")
    assert_parity(vg[:, :, sp:sp + S], vr, "bf16", "V cache (all written positions)")
    np.testing.assert_array_equal(kg[:, :, :sp], synth.as_f64(kc)[:, :, :sp])
    np.testing.assert_array_equal(kg[:, :, sp + S:], synth.as_f64(kc)[:, :, sp + S:])


def test_llama3_8b_decode_full_size():
    s = synth.SHAPES["llama3_8b_decode_b64"]
    B, S, sp = s["B"], s["S"], s["start_pos"]
    w = synth.block_weights(s)
    x = synth.block_activations(s)
    kc, vc = synth.kv_cache(s, fill_upto=sp)
    y, kg, vg = _run(s, w, x, kc, vc, B, S, sp)
    rows = [(b, 0) for b in range(B)]
    yr, kr, vr = oracle.block_forward_rows(s, f64_weights(w), synth.as_f64(x), sp, synth.as_f64(kc),
                                           synth.as_f64(vc), rows)
    assert_parity(y[:, 0], yr, "bf16", "y")
    assert_branch_parity(y[:, 0], yr, synth.as_f64(x)[:, 0], "y - x")
    assert_parity(kg[:, :, sp:sp + 1], kr, "bf16", "K cache slice")
    assert_parity(vg[:, :, sp:sp + 1], vr, "bf16", "V cache slice")
    np.testing.assert_array_equal(kg[:, :, :sp], synth.as_f64(kc)[:, :, :sp])


def test_chunked_prefill_then_decode_matches_oracle_chain():
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=96)
    B, L = 2, 96
    w = synth.block_weights(s)
    wf = f64_weights(w)
    x = synth.block_activations(s, tag="chain", B=B, S=70)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=L)
    t = torch()
    with GpuBlock(s, w, B * 64, max_seq_len=L) as blk:
        kd, vd = to_dev(kc), to_dev(vc)
        kr, vr = synth.as_f64(kc), synth.as_f64(vc)
        for (a, e) in [(0, 40), (40, 64), (64, 65), (65, 66), (66, 70)]:
            xs = np.ascontiguousarray(x[:, a:e])
            xd = to_dev(xs)
            yd = t.empty_like(xd)
            blk.lb.check(blk.forward(xd, yd, B, e - a, a, kd, vd))
            t.cuda.synchronize()
            yr, kr, vr = oracle.block_forward(s, wf, synth.as_f64(xs), a, kr, vr)
            assert_parity(to_f64(yd), yr, "bf16", f"chunk [{a}, {e})")
        assert_parity(to_f64(kd)[:, :, :70], kr[:, :, :70], "bf16", "K cache after the chain")


def test_y_may_alias_x_and_host_entry_point(lb):
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=40)
    B, S = 2, 40
    w = synth.block_weights(s)
    x = synth.block_activations(s, tag="alias", B=B, S=S)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=S)
    yr, _, _ = oracle.block_forward(s, f64_weights(w), synth.as_f64(x), 0, synth.as_f64(kc), synth.as_f64(vc))
    t = torch()
    with GpuBlock(s, w, B * S, max_seq_len=S) as blk:
        xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
        blk.lb.check(blk.forward(xd, xd, B, S, 0, kd, vd))
        t.cuda.synchronize()
        assert_parity(to_f64(xd), yr, "bf16", "y aliasing x")
        # host buffers: pinned in, pinned out, copies on the stream
        xh = t.from_numpy(x.view(np.int16)).view(t.bfloat16).pin_memory()
        yh = t.empty_like(xh).pin_memory()
        kd2, vd2 = to_dev(kc), to_dev(vc)
        kv = lb.make_kv_cache(kd2, vd2, B, S)
        stream = t.cuda.current_stream()
        lb.check(lb.llama_block_forward_host(blk.h, xh, yh, B, S, 0, kv, stream))
        stream.synchronize()
        assert_parity(to_f64(yh), yr, "bf16", "host-buffer entry point")


def test_forward_rejects_bad_calls_on_device(lb):
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=32)
    w = synth.block_weights(s)
    t = torch()
    with GpuBlock(s, w, 64, max_seq_len=32) as blk:
        kc = t.zeros((2, 3, 32, 64), dtype=t.bfloat16, device="cuda")
        vc = t.zeros_like(kc)
        x = t.zeros((2, 32, 576), dtype=t.bfloat16, device="cuda")
        y = t.empty_like(x)
        assert blk.forward(x, y, 3, 8, 0, kc, vc) == lb.LLAMA_ERR_RANGE        # B > max_batch
        assert blk.forward(x, y, 2, 8, 30, kc, vc) == lb.LLAMA_ERR_RANGE       # start_pos + S > max_seq
        assert blk.forward(x, y, 2, 40, 0, kc, vc) == lb.LLAMA_ERR_RANGE       # B*S > max_tokens
        assert blk.forward(x, y, 0, 8, 0, kc, vc) == lb.LLAMA_ERR_INVALID_ARG
        assert blk.forward(x, y, 1, 8, -1, kc, vc) == lb.LLAMA_ERR_INVALID_ARG
        xs = x.view(-1)[1:]  # 2-byte offset: misaligned
        assert blk.lb.llama_block_forward(blk.h, xs.data_ptr(), y, 1, 8, 0,
                                          lb.make_kv_cache(kc, vc, 2, 32), None) == lb.LLAMA_ERR_ALIGN
        xh = t.zeros((2, 32, 576), dtype=t.bfloat16)  # host memory passed as device pointer
        assert blk.forward(xh, y, 1, 8, 0, kc, vc) == lb.LLAMA_ERR_INVALID_ARG
        t.cuda.synchronize()
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_OK


def test_kernel_launch_count_per_forward(lb):
    """The bf16 path runs six kernels per prefill forward (row statistics, QKV+RoPE+cache, attention, O, gate/up,
    down) and seven per D=128 decode forward (the split-KV combine); the counter sees every one."""
    t = torch()
    for shape, B, S, start_pos, L, want in [
            (dict(synth.SHAPES["smollm2_135m"], max_seq_len=64), 2, 64, 0, 64, 6),
            (dict(synth.SHAPES["llama3_8b_decode_b64"], max_seq_len=600), 4, 1, 520, 600, 7)]:
        w = synth.block_weights(shape)
        with GpuBlock(shape, w, B * S, max_seq_len=L) as blk:
            G, D = shape["n_kv_heads"], shape["d_model"] // shape["n_heads"]
            kc = t.zeros((B, G, L, D), dtype=t.bfloat16, device="cuda")
            vc = t.zeros_like(kc)
            x = t.zeros((B, S, shape["d_model"]), dtype=t.bfloat16, device="cuda")
            y = t.empty_like(x)
            n0 = lb.llama_kernel_launch_count()
            lb.check(blk.forward(x, y, B, S, start_pos, kc, vc))
            assert lb.llama_kernel_launch_count() - n0 == want
            t.cuda.synchronize()
