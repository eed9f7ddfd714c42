"""Full-stack parity (embedding gather -> N blocks -> final RMSNorm -> untied LM
head) of llama_stack_forward against the fp64 oracle (GPU).

The stacks here are small enough for the oracle to finish in seconds: the tiny
fp32 model, a 30-layer SmolLM2-shaped model, and two Llama-3-8B-shaped layers
with a 32768-entry vocabulary (the per-layer work and the LM-head GEMM path
are the ones the 32-layer, 128256-vocabulary stack runs).  fp32 stacks and the
first layer's cache use the block bars; bf16 logits and deeper caches use the
stack bar derived in test_stack_tolerance.py.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import assert_parity, assert_stack_parity, make_cfg, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


def _stack_inputs(shape, n_layers, vocab, B, S, L):
    dt = shape["dtype"]
    layers = [synth.block_weights(shape, layer=l) for l in range(n_layers)]
    conv = (lambda a: a) if dt == "f32" else synth.f32_to_bf16_bits
    embed = conv(synth.normal(0, "embed", (vocab, shape["d_model"]), std=0.02))
    head = conv(synth.normal(0, "lm_head", (vocab, shape["d_model"]), std=0.02))
    fnorm = conv(synth.normal(0, "final_norm", (shape["d_model"],), std=0.1, mean=1.0))
    tokens = synth.uniform_int(0, "tokens", (B, S), vocab)
    caches = [synth.kv_cache(shape, max_batch=B, max_seq_len=L, layer=l) for l in range(n_layers)]
    return layers, embed, head, fnorm, tokens, caches


def _run_stack(lb, shape, layers, embed, head, fnorm, tokens, caches, B, S, start_pos, L):
    t = torch()
    wd = [{k: to_dev(v) for k, v in w.items()} for w in layers]
    st, stk = lb.llama_stack_create(make_cfg(shape, L), len(layers), embed.shape[0], to_dev(embed),
                                    [lb.make_weights(w) for w in wd], to_dev(fnorm), to_dev(head), B * S)
    lb.check(st, "llama_stack_create")
    try:
        kvd = [(to_dev(k), to_dev(v)) for k, v in caches]
        kvs = [lb.make_kv_cache(k, v, B, L) for k, v in kvd]
        tok = t.from_numpy(tokens).cuda()
        logits = t.empty((B, S, embed.shape[0]), dtype=t.float32, device="cuda")
        lb.check(lb.llama_stack_forward(stk, tok, B, S, start_pos, kvs, logits, t.cuda.current_stream()))
        t.cuda.synchronize()
        status = lb.llama_stack_device_status(stk)
        return logits.cpu().numpy().astype(np.float64), [(to_f64(k), to_f64(v)) for k, v in kvd], status
    finally:
        lb.llama_stack_destroy(stk)


def _oracle(shape, layers, embed, head, fnorm, tokens, caches, start_pos):
    return oracle.stack_forward(shape, [{k: synth.as_f64(v) for k, v in w.items()} for w in layers],
                                synth.as_f64(embed), synth.as_f64(fnorm), synth.as_f64(head), tokens, start_pos,
                                [(synth.as_f64(k), synth.as_f64(v)) for k, v in caches])


def test_tiny_f32_stack(lb):
    s = synth.SHAPES["tiny_f32"]
    B, S, L, vocab, n = 2, 8, 12, 50, 3
    args = _stack_inputs(s, n, vocab, B, S, L)
    logits, caches, status = _run_stack(lb, s, *args, B, S, 0, L)
    assert status == lb.LLAMA_OK
    ref, ref_caches = _oracle(s, *args, 0)
    assert_parity(logits, ref, "f32", "logits")
    for (kg, vg), (kr, vr) in zip(caches, ref_caches):
        assert_parity(kg[:, :, :S], kr[:, :, :S], "f32", "K cache")
        assert_parity(vg[:, :, :S], vr[:, :, :S], "f32", "V cache")


def test_stack_reports_out_of_range_token(lb):
    s = synth.SHAPES["tiny_f32"]
    B, S, L, vocab = 1, 4, 4, 50
    layers, embed, head, fnorm, tokens, caches = _stack_inputs(s, 1, vocab, B, S, L)
    tokens = tokens.copy()
    tokens[0, 2] = vocab + 7  # out of range: embedded as zeros and reported
    logits, _, status = _run_stack(lb, s, layers, embed, head, fnorm, tokens, caches, B, S, 0, L)
    assert status == lb.LLAMA_ERR_RANGE
    assert np.all(np.isfinite(logits))


def test_smollm2_30_layer_stack_bf16(lb):
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=64)
    B, S, L, vocab, n = 2, 48, 64, 49152, 30
    args = _stack_inputs(s, n, vocab, B, S, L)
    logits, caches, status = _run_stack(lb, s, *args, B, S, 0, L)
    assert status == lb.LLAMA_OK
    ref, ref_caches = _oracle(s, *args, 0)
    assert_stack_parity(logits, ref, "logits (30 layers)")
    assert_parity(caches[0][0][:, :, :S], ref_caches[0][0][:, :, :S], "bf16", "K cache layer 0")
    assert_parity(caches[0][1][:, :, :S], ref_caches[0][1][:, :, :S], "bf16", "V cache layer 0")
    assert_stack_parity(caches[n - 1][0][:, :, :S], ref_caches[n - 1][0][:, :, :S], f"K cache layer {n - 1}")
    assert_stack_parity(caches[n - 1][1][:, :, :S], ref_caches[n - 1][1][:, :, :S], f"V cache layer {n - 1}")


def test_llama3_8b_shaped_two_layer_stack_bf16(lb):
    s = dict(synth.SHAPES["llama3_8b_prefill_b1s8192"], max_seq_len=160)
    B, S, L, vocab, n = 1, 150, 160, 32768, 2
    args = _stack_inputs(s, n, vocab, B, S, L)
    logits, caches, status = _run_stack(lb, s, *args, B, S, 0, L)
    assert status == lb.LLAMA_OK
    ref, ref_caches = _oracle(s, *args, 0)
    assert_stack_parity(logits, ref, "logits (8B-shaped layers)")
    assert_parity(caches[0][0][:, :, :S], ref_caches[0][0][:, :, :S], "bf16", "K cache layer 0")
    assert_stack_parity(caches[1][0][:, :, :S], ref_caches[1][0][:, :, :S], "K cache layer 1")


def test_llama3_8b_shaped_three_layer_stack_on_cta_pairs_bf16(lb):
    """Three Llama-3-8B-shaped layers over a 2048-token prompt: every projection and the LM head
    (vocabulary 32768) run on CTA pairs, and the down projections' epilogues hand the next block's
    row statistics on through the alternating buffers."""
    s = dict(synth.SHAPES["llama3_8b_prefill_b1s8192"], max_seq_len=2048)
    B, S, L, vocab, n = 1, 2048, 2048, 32768, 3
    args = _stack_inputs(s, n, vocab, B, S, L)
    logits, caches, status = _run_stack(lb, s, *args, B, S, 0, L)
    assert status == lb.LLAMA_OK
    ref, ref_caches = _oracle(s, *args, 0)
    assert_stack_parity(logits, ref, "logits (8B-shaped layers, S=2048)")
    assert_parity(caches[0][0], ref_caches[0][0], "bf16", "K cache layer 0")
    assert_parity(caches[0][1], ref_caches[0][1], "bf16", "V cache layer 0")
    for l in (1, 2):
        assert_stack_parity(caches[l][0], ref_caches[l][0], f"K cache layer {l}")
        assert_stack_parity(caches[l][1], ref_caches[l][1], f"V cache layer {l}")


def test_odd_layer_stack_repeated_and_continued_through_one_handle_bf16(lb):
    """A bf16 stack hands each block's row statistics to the next through two
    alternating buffers that the consuming epilogues clear.  With an odd layer
    count the buffers end a forward in a different state than they start it, so
    one handle runs the same prefill twice and then a one-token step per
    sequence, each against the oracle."""
    t = torch()
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=64)
    B, S, L, vocab, n = 2, 40, 64, 4096, 3
    layers, embed, head, fnorm, tokens, caches = _stack_inputs(s, n, vocab, B, S, L)
    nxt = synth.uniform_int(0, "next_tokens", (B, 1), vocab)
    ref, ref_caches = _oracle(s, layers, embed, head, fnorm, tokens, caches, 0)
    ref2, _ = _oracle(s, layers, embed, head, fnorm, nxt, ref_caches, S)
    wd = [{k: to_dev(v) for k, v in w.items()} for w in layers]
    st, stk = lb.llama_stack_create(make_cfg(s, L), n, vocab, to_dev(embed), [lb.make_weights(w) for w in wd],
                                    to_dev(fnorm), to_dev(head), B * S)
    lb.check(st, "llama_stack_create")
    try:
        kvd = [(to_dev(k), to_dev(v)) for k, v in caches]
        kvs = [lb.make_kv_cache(k, v, B, L) for k, v in kvd]
        stream = t.cuda.current_stream()
        tok = t.from_numpy(tokens).cuda()
        for rep in range(2):
            logits = t.empty((B, S, vocab), dtype=t.float32, device="cuda")
            lb.check(lb.llama_stack_forward(stk, tok, B, S, 0, kvs, logits, stream))
            t.cuda.synchronize()
            assert lb.llama_stack_device_status(stk) == lb.LLAMA_OK
            assert_stack_parity(logits.cpu().numpy().astype(np.float64), ref, f"prefill logits, forward {rep + 1}")
        logits = t.empty((B, 1, vocab), dtype=t.float32, device="cuda")
        lb.check(lb.llama_stack_forward(stk, t.from_numpy(nxt).cuda(), B, 1, S, kvs, logits, stream))
        t.cuda.synchronize()
        assert lb.llama_stack_device_status(stk) == lb.LLAMA_OK
        assert_stack_parity(logits.cpu().numpy().astype(np.float64), ref2, "one-token step logits")
    finally:
        lb.llama_stack_destroy(stk)
