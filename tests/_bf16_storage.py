"""A model of where a bf16 tensor-core block stores values (CPU, test-side).

The library's bf16 path rounds to bf16 exactly where it stores a value: the
RMSNorm gains folded into the weights they feed (bf16(W * g), once at create
time -- the normalised activations are never stored, the row scale is applied
to the fp32 accumulator), q and k after RoPE and v (one rounding each, from the
fp32 accumulator), P before the PV product, the attention output o, the SwiGLU
product, and the residual stream h and y.  `block` replays the oracle's exact
arithmetic (oracle.rope, exact softmax, fp64 products) with a bf16 rounding at
each of those points.  It is a model of the storage precision, not of any
kernel: it fixes how far a correct bf16 implementation must land from the
exact fp64 oracle, which sets the parity bar of deep stacks.

residual_f32=True models the alternative of keeping the residual stream (h
and y) in fp32 between the branches and blocks: the GEMM operands are then
bf16 copies of it, the row statistics come from the fp32 values.
"""
import math

import numpy as np

import oracle
import synth


def bf(a):
    """fp64 -> nearest bf16 (via fp32) -> fp64."""
    return synth.as_f64(synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32)))


def block(cfg, w, x, start_pos=0, residual_f32=False):
    """One block with start_pos = 0 and an empty cache.  x: [B, S, d] (fp64
    values).  Returns (y, k, v): the block output and the cached K (rotated)
    and V, [B, S, G, D], as the model stores them."""
    assert start_pos == 0
    d, H, G = cfg["d_model"], cfg["n_heads"], cfg["n_kv_heads"]
    D, r = d // H, H // G
    B, S, _ = x.shape
    eps = cfg["norm_eps"]
    res = (lambda a: a) if residual_f32 else bf
    xa = bf(x)  # the GEMM operand (x itself when the stream is bf16)
    rs = 1.0 / np.sqrt(np.mean(x * x, -1, keepdims=True) + eps)  # row scale, applied after the GEMM
    g1 = w["attn_norm"]
    pos = np.arange(S)
    q = bf(oracle.rope((rs * (xa @ bf(w["wq"] * g1).T)).reshape(B, S, H, D), pos, cfg["rope_theta"]))
    k = bf(oracle.rope((rs * (xa @ bf(w["wk"] * g1).T)).reshape(B, S, G, D), pos, cfg["rope_theta"]))
    v = bf(rs * (xa @ bf(w["wv"] * g1).T)).reshape(B, S, G, D)
    o = np.zeros((B, S, H, D))
    vis = np.arange(S)[None, :] <= np.arange(S)[:, None]
    for b in range(B):
        for h in range(H):
            sc = np.where(vis, q[b, :, h] @ k[b, :, h // r].T / math.sqrt(D), -np.inf)
            p = np.exp(sc - sc.max(-1, keepdims=True))
            o[b, :, h] = (bf(p) @ v[b, :, h // r]) / p.sum(-1, keepdims=True)
    hres = res(x + bf(o.reshape(B, S, H * D)) @ w["wo"].T)
    ha = bf(hres)
    rs2 = 1.0 / np.sqrt(np.mean(hres * hres, -1, keepdims=True) + eps)
    g2 = w["ffn_norm"]
    gt, up = rs2 * (ha @ bf(w["w_gate"] * g2).T), rs2 * (ha @ bf(w["w_up"] * g2).T)
    y = res(hres + bf(gt / (1 + np.exp(-gt)) * up) @ w["w_down"].T)
    return y, k, v


def logits(cfg, x, final_norm, lm_head):
    """Final RMSNorm (rounded once, to the head GEMM's bf16 operand) and the
    fp32-output LM head."""
    return bf(oracle.rms_norm(x, final_norm, cfg["norm_eps"])) @ lm_head.T
