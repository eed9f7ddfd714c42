"""Mixture-of-experts blocks against the fp64 oracle (GPU).

Routing is an arg-max taken in floating point: where two router logits are
closer than the rounding of the bf16 path, either choice is correct.  So the
test
- checks that every expert the GPU chose is a top-k choice of the oracle's
  router logits within a bar (and that each token's choices are distinct),
- evaluates the oracle block on the GPU's choice of experts (their weights
  recomputed by the oracle, in fp64), and compares y and the cache with the
  bf16 parity bars.
Shapes cover single and multi-tile experts, experts that receive no row, a
shared expert and none, prefill and decode.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import GpuBlock, assert_branch_parity, assert_parity, f64_weights, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu

BASE = dict(norm_eps=1e-5, dtype="bf16", max_seq_len=256)
MOE_SHAPES = {
    # d, heads, experts, top k, expert width, shared width
    "small_shared": dict(BASE, d_model=256, n_heads=4, n_kv_heads=2, rope_theta=1e4, d_ff=128, n_experts=8, top_k=2,
                         d_ff_shared=256),
    "d128_heads_shared": dict(BASE, d_model=1024, n_heads=8, n_kv_heads=2, rope_theta=5e5, d_ff=512, n_experts=16,
                              top_k=2, d_ff_shared=1024),
    "many_experts_no_shared": dict(BASE, d_model=512, n_heads=8, n_kv_heads=4, rope_theta=1e5, d_ff=256,
                                   n_experts=64, top_k=4, d_ff_shared=0),
    "few_experts_multi_tile": dict(BASE, d_model=512, n_heads=4, n_kv_heads=4, rope_theta=1e4, d_ff=384, n_experts=4,
                                   top_k=2, d_ff_shared=0),
}


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


def _run_moe(lb, shape, B, S, start_pos, L, fill_upto, tag):
    t = torch()
    w = synth.block_weights(shape)
    x = synth.block_activations(shape, tag=tag, B=B, S=S)
    kc, vc = synth.kv_cache(shape, max_batch=B, max_seq_len=L, fill_upto=fill_upto)
    k = shape["top_k"]
    with GpuBlock(shape, w, B * S, max_seq_len=L) as blk:
        xd, kd, vd = to_dev(x), to_dev(kc), to_dev(vc)
        yd = t.empty_like(xd)
        lb.check(blk.forward(xd, yd, B, S, start_pos, kd, vd), "llama_block_forward")
        ids = t.empty((B * S, k), dtype=t.int32, device="cuda")
        wts = t.empty((B * S, k), dtype=t.float32, device="cuda")
        lb.check(lb.llama_block_moe_routing(blk.h, ids, wts, t.cuda.current_stream()), "routing")
        t.cuda.synchronize()
        assert lb.llama_block_device_status(blk.h) == lb.LLAMA_OK
        return (w, x, kc, vc, to_f64(yd), to_f64(kd), to_f64(vd), ids.cpu().numpy().astype(np.int64),
                wts.cpu().numpy().astype(np.float64))


def _check(shape, B, S, start_pos, L, fill_upto, tag, lb):
    w, x, kc, vc, y, kg, vg, ids, wts = _run_moe(lb, shape, B, S, start_pos, L, fill_upto, tag)
    wf = f64_weights(w)
    k = shape["top_k"]
    h, _, _ = oracle.block_residual_h(shape, wf, synth.as_f64(x), start_pos, synth.as_f64(kc), synth.as_f64(vc))
    v = oracle.rms_norm(h, wf["ffn_norm"], shape["norm_eps"]).reshape(B * S, -1)
    _, _, logits = oracle.moe_route(shape, wf, v)
    # each GPU choice is a top-k choice of the oracle's logits within the bar; choices are distinct
    kth = -np.sort(-logits, axis=-1)[:, k - 1]
    bar = 2e-2 * np.max(np.abs(logits), axis=-1) + 1e-3
    chosen = np.take_along_axis(logits, ids, -1)
    assert np.all((ids >= 0) & (ids < shape["n_experts"]))
    assert all(len(set(r)) == k for r in ids.tolist())
    assert np.all(chosen >= kth[:, None] - bar[:, None]), "a GPU-chosen expert is not a top-k choice"
    # weights: softmax over the chosen logits, by the oracle
    e = np.exp(chosen - chosen.max(-1, keepdims=True))
    w_ref = e / e.sum(-1, keepdims=True)
    np.testing.assert_allclose(wts, w_ref, rtol=0, atol=1e-2)
    np.testing.assert_allclose(wts.sum(-1), 1.0, rtol=0, atol=1e-5)
    # the block output on the GPU's routing decision
    yr, kr, vr = oracle.block_forward(shape, wf, synth.as_f64(x), start_pos, synth.as_f64(kc), synth.as_f64(vc),
                                      route=(ids, w_ref))
    assert_parity(y, yr, "bf16", "y")
    assert_branch_parity(y, yr, synth.as_f64(x), "y - x (both branch outputs)")
    sl = (slice(0, B), slice(None), slice(start_pos, start_pos + S))
    assert_parity(kg[sl], kr[sl], "bf16", "K cache slice")
    assert_parity(vg[sl], vr[sl], "bf16", "V cache slice")
    return ids


@pytest.mark.parametrize("name", list(MOE_SHAPES))
def test_moe_block_prefill(lb, name):
    shape = MOE_SHAPES[name]
    B, S = (2, 300) if name == "few_experts_multi_tile" else (2, 40)
    ids = _check(shape, B, S, 0, S + 8, 0, "moe_" + name, lb)
    if name == "few_experts_multi_tile":  # some expert received more than one 128-row tile
        assert np.bincount(ids.ravel(), minlength=shape["n_experts"]).max() > 128


def test_moe_block_prefill_on_cta_pairs(lb):
    """8192 routed rows (4096 tokens, top-2 of 8 experts): the experts' grouped GEMMs run 256-row tiles
    per expert on CTA pairs (rows past an expert's range inside a tile are computed and not stored),
    and so do the shared expert's GEMMs."""
    shape = dict(BASE, d_model=1024, n_heads=8, n_kv_heads=2, rope_theta=5e5, d_ff=1024, n_experts=8, top_k=2,
                 d_ff_shared=1024, max_seq_len=2048)
    B, S = 2, 2048
    ids = _check(shape, B, S, 0, S, 0, "moe_pairs", lb)
    counts = np.bincount(ids.ravel(), minlength=shape["n_experts"])
    assert counts.sum() == B * S * 2 and counts.max() > 512  # experts span several 256-row tiles


@pytest.mark.parametrize("name", ["small_shared", "d128_heads_shared"])
def test_moe_block_decode(lb, name):
    _check(MOE_SHAPES[name], 4, 1, 37, 48, 37, "moe_dec_" + name, lb)


def test_moe_experts_without_rows(lb):
    shape = MOE_SHAPES["many_experts_no_shared"]
    ids = _check(shape, 1, 6, 0, 8, 0, "moe_sparse", lb)  # 24 choices over 64 experts
    assert np.bincount(ids.ravel(), minlength=64).min() == 0


def test_moe_routing_is_rejected_for_dense_blocks(lb):
    t = torch()
    shape = dict(synth.SHAPES["smollm2_135m"], max_seq_len=16)
    with GpuBlock(shape, synth.block_weights(shape), 8, max_seq_len=16) as blk:
        ids = t.empty((8, 2), dtype=t.int32, device="cuda")
        wts = t.empty((8, 2), dtype=t.float32, device="cuda")
        assert lb.llama_block_moe_routing(blk.h, ids, wts, None) == lb.LLAMA_ERR_INVALID_ARG
