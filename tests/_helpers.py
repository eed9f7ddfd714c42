"""Shared helpers of the GPU parity tests: marshalling synth arrays to torch
device tensors, running the library, and the parity criteria."""
from __future__ import annotations

import numpy as np

import synth

# Parity bars (fp32: max|err| <= 1e-4 max|ref|; bf16 with fp32 accumulation:
# relative Frobenius <= 5e-3 and max|err| <= 3e-2 max|ref|).
F32_MAX_REL = 1e-4
BF16_FRO_REL = 5e-3
BF16_MAX_REL = 3e-2


def torch():
    import torch as _t
    return _t


def to_dev(a: np.ndarray):
    t = torch()
    if a.dtype == np.uint16:
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host_bits(tensor) -> np.ndarray:
    """Stored representation on the host: uint16 bf16 bits, or fp32/int32 as is."""
    t = torch()
    c = tensor.detach().cpu().contiguous()
    if c.dtype == t.bfloat16:
        return c.view(t.int16).numpy().view(np.uint16)
    return c.numpy()


def to_f64(tensor) -> np.ndarray:
    return synth.as_f64(to_host_bits(tensor))


def parity_errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    fro = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(diff)) / max(np.max(np.abs(ref)), 1e-300)) if ref.size else 0.0
    return fro, mx


def assert_parity(got, ref, dtype: str, what: str):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    fro, mx = parity_errors(got, ref)
    if dtype == "f32":
        assert mx <= F32_MAX_REL, f"{what}: max|err|/max|ref| = {mx:.3e} > {F32_MAX_REL}"
    else:
        assert fro <= BF16_FRO_REL and mx <= BF16_MAX_REL, (
            f"{what}: rel-Frobenius {fro:.3e} (bar {BF16_FRO_REL}), max|err|/max|ref| {mx:.3e} (bar {BF16_MAX_REL})")
    return fro, mx


# Relative-Frobenius bar for the logits (and deep-layer caches) of a multi-layer
# bf16 stack: storing every GEMM operand in bf16 already moves two
# Llama-3-8B-shaped layers ~1.2 % from the exact result (derived and pinned in
# test_stack_tolerance.py); the bar keeps a factor two above that.
STACK_FRO_REL = 2.5e-2


def assert_stack_parity(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    fro, mx = parity_errors(got, ref)
    assert fro <= STACK_FRO_REL and mx <= BF16_MAX_REL, (
        f"{what}: rel-Frobenius {fro:.3e} (bar {STACK_FRO_REL}), max|err|/max|ref| {mx:.3e} (bar {BF16_MAX_REL})")
    return fro, mx


def bf16_round(a: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 (via fp32) -> fp64."""
    return synth.as_f64(synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32)))


def assert_branch_parity(y_got, y_ref, x, what):
    """Parity of the summed branch outputs y - x of a bf16 block.

    y is stored in bf16, so (y - x) carries y's own output rounding (and that of
    the bf16 h stored between the branches) on top of the branch arithmetic.
    Bar: ||err|| <= 5e-3 ||y_ref - x|| + 2 ||bf16(y_ref) - y_ref||, i.e. the bf16
    relative-Frobenius bar on the branches plus twice the unavoidable rounding
    of one bf16 store of y (measured on the reference itself)."""
    y_got = np.asarray(y_got, dtype=np.float64)
    ref_b = np.asarray(y_ref, dtype=np.float64) - x
    err = float(np.linalg.norm((y_got - x) - ref_b))
    round_err = float(np.linalg.norm(bf16_round(y_ref) - y_ref))
    bar = BF16_FRO_REL * float(np.linalg.norm(ref_b)) + 2.0 * round_err
    assert err <= bar, f"{what}: ||err|| {err:.4e} > bar {bar:.4e} (rounding part {2 * round_err:.4e})"
    return err, bar


def llama_dtype(shape):
    import decoder_block_gb300 as lb
    return lb.LLAMA_BF16 if shape["dtype"] == "bf16" else lb.LLAMA_F32


def make_cfg(shape, max_seq_len=None):
    import decoder_block_gb300 as lb
    layout = {"interleaved": lb.LLAMA_ROPE_INTERLEAVED, "halves": lb.LLAMA_ROPE_HALVES}[
        shape.get("rope_layout", "interleaved")]
    return lb.make_config(shape["d_model"], shape["n_heads"], shape["n_kv_heads"], shape["d_ff"],
                          max_seq_len or shape["max_seq_len"], shape["norm_eps"], shape["rope_theta"],
                          llama_dtype(shape), layout, shape.get("rope_scaling"), shape.get("n_experts", 0),
                          shape.get("top_k", 0), shape.get("d_ff_shared", 0))


def f64_weights(w: dict) -> dict:
    return {k: synth.as_f64(v) for k, v in w.items()}


class GpuBlock:
    """One library block handle with device copies of the weights."""

    def __init__(self, shape, w_np: dict, max_tokens: int, max_seq_len=None):
        import decoder_block_gb300 as lb
        self.lb = lb
        self.shape = shape
        self.w_dev = {k: to_dev(v) for k, v in w_np.items()}
        st, self.h = lb.llama_block_create(make_cfg(shape, max_seq_len), lb.make_weights(self.w_dev), max_tokens)
        lb.check(st, "llama_block_create")

    def forward(self, x_dev, y_dev, B, S, start_pos, kc_dev, vc_dev, stream=None):
        lb = self.lb
        kv = lb.make_kv_cache(kc_dev, vc_dev, kc_dev.shape[0], kc_dev.shape[2])
        st = lb.llama_block_forward(self.h, x_dev, y_dev, B, S, start_pos, kv,
                                    stream if stream is not None else torch().cuda.current_stream())
        return st

    def close(self):
        if self.h:
            self.lb.llama_block_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()
