"""Failure detection by bounded waits, made to run out on the GPU.

Every wait of the library's kernels that can give up is bounded by the
handle's wait budget (about 2 s by default).  Here a SmolLM2-shaped block
(B = 8, S = 1024: every GEMM runs whole output tiles) gets a one-cycle budget,
so the first wait of each tensor-core kernel that is not satisfied at once
gives up: the kernel records the timeout in the handle's status word, its
other roles give up too, and it returns once the copies and MMAs it had issued
have landed and its tensor memory is freed.  The test checks that the host
reads LLAMA_ERR_DEVICE_TIMEOUT (once: reading clears it), that the CUDA
context is still usable, and that the same handle with the default budget, and
a fresh handle, then match the fp64 oracle.  A Llama-3-8B-shaped prefill
does the same through the GEMMs that run on CTA pairs.  Nothing here faults
or traps.
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


def _forward(blk, x, kc, vc, B, S):
    t = torch()
    xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
    yd = t.full_like(xd, float("nan"))
    blk.lb.check(blk.forward(xd, yd, B, S, 0, kd, vd), "llama_block_forward")
    t.cuda.synchronize()  # raises if a kernel faulted: none may
    return yd, kd, vd


def _check(lb, blk, s, x, ref, B, S, what):
    yd, kd, vd = _forward(blk, x, *ref["caches"], B, S)
    assert lb.llama_block_device_status(blk.h) == lb.LLAMA_OK, what
    y = to_f64(yd)
    assert_parity(y, ref["y"], "bf16", f"{what}: y")
    assert_branch_parity(y, ref["y"], synth.as_f64(x), f"{what}: y - x")
    assert_parity(to_f64(kd)[:, :, :S], ref["k"][:, :, :S], "bf16", f"{what}: K cache")
    assert_parity(to_f64(vd)[:, :, :S], ref["v"][:, :, :S], "bf16", f"{what}: V cache")


def test_wait_that_runs_out_is_reported_and_the_context_recovers(lb):
    s = synth.SHAPES["smollm2_135m"]
    B, S = s["B"], s["S"]
    w = synth.block_weights(s)
    x = synth.block_activations(s, B=B, S=S)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=S)
    yr, kr, vr = oracle.block_forward(s, f64_weights(w), synth.as_f64(x), 0, synth.as_f64(kc), synth.as_f64(vc))
    ref = {"y": yr, "k": kr, "v": vr, "caches": (kc, vc)}

    with GpuBlock(s, w, B * S) as blk:
        assert lb.llama_block_set_wait_budget(blk.h, -1) == lb.LLAMA_ERR_INVALID_ARG
        assert lb.llama_block_set_wait_budget(None, 0) == lb.LLAMA_ERR_INVALID_ARG
        lb.check(lb.llama_block_set_wait_budget(blk.h, 1), "set a one-cycle wait budget")
        _forward(blk, x, kc, vc, B, S)
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_ERR_DEVICE_TIMEOUT
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_OK  # the read cleared it
        # the same handle, back on the default budget
        lb.check(lb.llama_block_set_wait_budget(blk.h, 0), "restore the default budget")
        _check(lb, blk, s, x, ref, B, S, "same handle after the timeout")

    with GpuBlock(s, w, B * S) as fresh:
        _check(lb, fresh, s, x, ref, B, S, "fresh handle")


def test_stack_wait_budget_setter(lb):
    s = synth.SHAPES["tiny_f32"]
    t = torch()
    w = {k: to_dev(v) for k, v in synth.block_weights(s).items()}
    emb = to_dev(synth.normal(0, "embed", (50, s["d_model"]), std=0.02))
    head = to_dev(synth.normal(0, "lm_head", (50, s["d_model"]), std=0.02))
    fn = to_dev(synth.normal(0, "final_norm", (s["d_model"],), std=0.1, mean=1.0))
    from _helpers import make_cfg
    st, stk = lb.llama_stack_create(make_cfg(s), 1, 50, emb, [lb.make_weights(w)], fn, head, 16)
    lb.check(st, "llama_stack_create")
    try:
        assert lb.llama_stack_set_wait_budget(stk, -5) == lb.LLAMA_ERR_INVALID_ARG
        lb.check(lb.llama_stack_set_wait_budget(stk, 1000000), "set")
        lb.check(lb.llama_stack_set_wait_budget(stk, 0), "reset")
        assert lb.llama_stack_device_status(stk) == lb.LLAMA_OK
        t.cuda.synchronize()
    finally:
        lb.llama_stack_destroy(stk)


def test_wait_that_runs_out_in_cta_pair_gemms(lb):
    """The same on a Llama-3-8B-shaped prefill (B = 1, S = 2048), whose four
    GEMMs run as 256 x 256 tiles on CTA pairs: a wait that gives up in one CTA
    of a pair makes its peer give up too, the pair settles the copies either
    producer issued before both leave, and the handle recovers."""
    s = dict(synth.SHAPES["llama3_8b_prefill_b4s2048"], B=1)
    B, S = 1, 2048
    w = synth.block_weights(s)
    x = synth.block_activations(s, B=B, S=S)
    kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=S)
    rows = [(0, 0), (0, 127), (0, 128), (0, 255), (0, 256), (0, 1023), (0, 2047)]
    yr, kr, vr = oracle.block_forward_rows(s, f64_weights(w), synth.as_f64(x), 0, synth.as_f64(kc),
                                           synth.as_f64(vc), rows)
    with GpuBlock(s, w, B * S) as blk:
        lb.check(lb.llama_block_set_wait_budget(blk.h, 1), "set a one-cycle wait budget")
        _forward(blk, x, kc, vc, B, S)
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_ERR_DEVICE_TIMEOUT
        lb.check(lb.llama_block_set_wait_budget(blk.h, 0), "restore the default budget")
        yd, kd, vd = _forward(blk, x, kc, vc, B, S)
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_OK
    y = to_f64(yd)
    ys = np.stack([y[b, t] for b, t in rows])
    assert_parity(ys, yr, "bf16", "y (sampled rows) after the timeout")
    assert_parity(to_f64(kd)[:, :, :S], kr, "bf16", "K cache after the timeout")
    assert_parity(to_f64(vd)[:, :, :S], vr, "bf16", "V cache after the timeout")
