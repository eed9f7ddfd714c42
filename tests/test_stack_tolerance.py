"""Derivation of the stack-logits tolerance (CPU).

A bf16 tensor-core stack rounds values to bf16 wherever it stores them (the
points are listed in _bf16_storage.py).  Replaying the oracle's exact
arithmetic with a bf16 rounding at each of those points (a model of the
storage precision, not of any kernel) shows how far a correct bf16 stack's
logits land from the exact fp64 oracle.  For two Llama-3-8B-shaped layers that
inherent error is about 1 % relative Frobenius -- above the 5e-3 bar that holds
for a single block -- so multi-layer stacks of up to a few layers are compared
with STACK_LOGITS_FRO_REL = 2.5e-2, at least twice the emulated error; the
max-error bar (3e-2 max|ref|) is unchanged.  Keeping the residual stream in
fp32 between the branches and blocks does not bring the error under 5e-3
either: the rounding of the GEMM operands, of the folded weights, of q, k, v,
P and of the SwiGLU product is what carries it.  Deeper stacks (the 32-layer
8B stack) take their bar from the same model evaluated at their own depth
(test_stack_8b_gpu.py).
"""
import numpy as np

import _bf16_storage as bfs
import oracle
import synth

STACK_LOGITS_FRO_REL = 2.5e-2


def _two_layer_8b(residual_f32):
    s = dict(synth.SHAPES["llama3_8b_prefill_b1s8192"], max_seq_len=40)
    B, S, vocab, n = 1, 40, 2048, 2
    layers = [{k: synth.as_f64(v) for k, v in synth.block_weights(s, layer=l).items()} for l in range(n)]
    embed = bfs.bf(synth.normal(0, "embed", (vocab, s["d_model"]), std=0.02))
    head = bfs.bf(synth.normal(0, "lm_head", (vocab, s["d_model"]), std=0.02))
    fnorm = bfs.bf(synth.normal(0, "final_norm", (s["d_model"],), std=0.1, mean=1.0))
    tokens = synth.uniform_int(0, "tokens", (B, S), vocab)
    kc = np.zeros((B, s["n_kv_heads"], S, s["d_model"] // s["n_heads"]))
    ref, _ = oracle.stack_forward(s, layers, embed, fnorm, head, tokens, 0, [(kc, kc)] * n)
    out = {}
    for mode in residual_f32:
        x = embed[tokens]
        for w in layers:
            x, _, _ = bfs.block(s, w, x, residual_f32=mode)
        emu = bfs.logits(s, x, fnorm, head)
        out[mode] = (float(np.linalg.norm(emu - ref) / np.linalg.norm(ref)),
                     float(np.max(np.abs(emu - ref)) / np.max(np.abs(ref))))
    return out


def test_bf16_storage_error_of_a_two_layer_8b_stack_sets_the_logits_bar():
    errs = _two_layer_8b((False, True))
    err, mx = errs[False]
    err32, _ = errs[True]
    print(f"emulated bf16-storage logits error: {err:.3e} relative Frobenius "
          f"({err32:.3e} with an fp32 residual stream)")
    # the storage precision alone exceeds the single-block bar ...
    assert err > 5e-3
    # ... an fp32 residual stream does not change that ...
    assert err32 > 5e-3
    # ... and the stack bar leaves at least a factor two above it
    assert 2.0 * err <= STACK_LOGITS_FRO_REL
    assert mx < 3e-2
