"""Greedy decoding through the stack (llama_stack_generate) against the fp64
oracle (GPU).

Two kinds of check:
- a model whose answer is unique by construction (one-hot embeddings, blocks
  whose output projections vanish, a permutation LM head): the generated ids
  must equal the closed-form chain exactly;
- random stacks, where near-equal logits can legitimately flip an arg-max:
  every id the GPU picks must be a maximum of the oracle's logits (teacher
  forced on the GPU's own history) within the parity bar, the last step's
  logits must meet the stack bar, and the returned ids must be the exact
  arg-max of the returned logits.
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


def _conv(dt, a):
    return np.asarray(a, dtype=np.float32) if dt == "f32" else synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def _generate(lb, shape, layers, embed, head, fnorm, prompt, start_pos, n_new, L, fill=0.0):
    t = torch()
    dt = shape["dtype"]
    B, S = prompt.shape
    vocab = embed.shape[0]
    G, D = shape["n_kv_heads"], shape["d_model"] // shape["n_heads"]
    wd = [{k: to_dev(v) for k, v in w.items()} for w in layers]
    st, stk = lb.llama_stack_create(make_cfg(shape, L), len(layers), vocab, to_dev(embed),
                                    [lb.make_weights(w) for w in wd], to_dev(fnorm), to_dev(head), B * S)
    lb.check(st, "llama_stack_create")
    try:
        tdt = t.float32 if dt == "f32" else t.bfloat16
        caches = [(t.full((B, G, L, D), fill, dtype=tdt, device="cuda"), t.full((B, G, L, D), fill, dtype=tdt,
                                                                             device="cuda")) for _ in layers]
        kvs = [lb.make_kv_cache(k, v, B, L) for k, v in caches]
        tok = t.from_numpy(prompt.astype(np.int32)).cuda()
        out = t.full((B, n_new), -1, dtype=t.int32, device="cuda")
        logits = t.empty((B, vocab), dtype=t.float32, device="cuda")
        lb.check(lb.llama_stack_generate(stk, tok, B, S, start_pos, n_new, kvs, out, logits,
                                         t.cuda.current_stream()), "llama_stack_generate")
        t.cuda.synchronize()
        assert lb.llama_stack_device_status(stk) == lb.LLAMA_OK
        return (out.cpu().numpy().astype(np.int64), logits.cpu().numpy().astype(np.float64),
                [(to_f64(k), to_f64(v)) for k, v in caches])
    finally:
        lb.llama_stack_destroy(stk)


def _identity_layers(shape, n, dt):
    layers = []
    for l in range(n):
        w = synth.block_weights(shape, layer=l)
        w["wo"] = np.zeros_like(w["wo"])
        w["w_down"] = np.zeros_like(w["w_down"])
        layers.append(w)
    return layers


@pytest.mark.parametrize("name", ["tiny_f32", "smollm2_135m"])
def test_generate_follows_the_closed_form_chain_exactly(lb, name):
    shape = synth.SHAPES[name]
    dt, d = shape["dtype"], shape["d_model"]
    vocab = min(d, 61)
    perm = synth.uniform_int(0, "gen/perm", (vocab,), 1 << 30).argsort()
    inv = np.argsort(perm)
    emb = np.zeros((vocab, d), np.float32)
    emb[np.arange(vocab), np.arange(vocab)] = 3.0
    head = np.zeros((vocab, d), np.float32)
    head[np.arange(vocab), perm] = 1.0
    prompt = synth.uniform_int(0, "gen/prompt", (3, 5), vocab)
    start_pos, n_new, L = 2, 7, 16
    layers = _identity_layers(shape, 2, dt)
    toks, last, caches = _generate(lb, shape, layers, _conv(dt, emb), _conv(dt, head), _conv(dt, np.ones(d)),
                                   prompt, start_pos, n_new, L, fill=7.0)
    want = np.zeros_like(toks)
    for b in range(3):
        t = prompt[b, -1]
        for i in range(n_new):
            t = inv[t]
            want[b, i] = t
    np.testing.assert_array_equal(toks, want)
    np.testing.assert_array_equal(np.argmax(last, -1), toks[:, -1])
    # positions start_pos .. start_pos + S + n_new - 2 are written, every other one keeps its fill
    hi = start_pos + prompt.shape[1] + n_new - 1
    for kc, vc in caches:
        assert np.all(kc[:, :, :start_pos] == 7.0) and np.all(kc[:, :, hi:] == 7.0)
        assert np.all(vc[:, :, :start_pos] == 7.0) and np.all(vc[:, :, hi:] == 7.0)
        assert not np.any(np.all(kc[:, :, start_pos:hi] == 7.0, axis=-1))


def _check_against_oracle(shape, layers, emb, head, fnorm, prompt, start_pos, toks, last, L, dt):
    """Teacher-forced oracle logits over the GPU's own history: each picked id is a maximum within the bar."""
    B, S = prompt.shape
    n_new = toks.shape[1]
    G, D = shape["n_kv_heads"], shape["d_model"] // shape["n_heads"]
    f64 = [{k: synth.as_f64(v) for k, v in w.items()} for w in layers]
    fresh = [(np.zeros((B, G, L, D)), np.zeros((B, G, L, D))) for _ in layers]
    seq = np.concatenate([prompt, toks[:, :-1]], 1)
    ref, _ = oracle.stack_forward(shape, f64, synth.as_f64(emb), synth.as_f64(fnorm), synth.as_f64(head), seq,
                                  start_pos, fresh)
    ref = ref[:, S - 1:]  # the logits that choose toks[:, i]
    bar = 2.0 * (1e-4 if dt == "f32" else 3e-2)
    for b in range(B):
        for i in range(n_new):
            row = ref[b, i]
            assert row[toks[b, i]] >= row.max() - bar * np.max(np.abs(row)), (b, i)
    np.testing.assert_array_equal(np.argmax(last, -1), toks[:, -1])
    if dt == "f32":
        assert_parity(last, ref[:, -1], "f32", "last-step logits")
    else:
        assert_stack_parity(last, ref[:, -1], "last-step logits")
    return ref


def test_generate_tiny_f32_stack_matches_oracle(lb):
    shape = synth.SHAPES["tiny_f32"]
    vocab, B, S, n_new, L, start_pos = 50, 2, 6, 5, 16, 1
    layers = [synth.block_weights(shape, layer=l) for l in range(3)]
    emb = synth.normal(0, "gen/embed", (vocab, shape["d_model"]), std=1.0)
    head = synth.normal(0, "gen/head", (vocab, shape["d_model"]), std=0.3)
    fnorm = synth.normal(0, "gen/fnorm", (shape["d_model"],), std=0.1, mean=1.0)
    prompt = synth.uniform_int(0, "gen/tiny_prompt", (B, S), vocab)
    toks, last, _ = _generate(lb, shape, layers, emb, head, fnorm, prompt, start_pos, n_new, L)
    ref = _check_against_oracle(shape, layers, emb, head, fnorm, prompt, start_pos, toks, last, L, "f32")
    # the oracle's own greedy chain agrees wherever its top-2 margin is clear
    want, _, _ = oracle.greedy_generate(shape, [{k: synth.as_f64(v) for k, v in w.items()} for w in layers],
                                        synth.as_f64(emb), synth.as_f64(fnorm), synth.as_f64(head), prompt,
                                        start_pos,
                                        [(np.zeros((B, 2, L, 16)), np.zeros((B, 2, L, 16))) for _ in layers], n_new)
    top2 = np.sort(ref, -1)[..., -2:]
    if np.all(top2[..., 1] - top2[..., 0] > 1e-3 * np.abs(ref).max()):
        np.testing.assert_array_equal(toks, want)


def test_generate_llama3_8b_shaped_two_layers_bf16(lb):
    shape = dict(synth.SHAPES["llama3_8b_prefill_b1s8192"], max_seq_len=64)
    vocab, B, S, n_new, L = 32768, 2, 16, 4, 64
    layers = [synth.block_weights(shape, layer=l) for l in range(2)]
    emb = synth.f32_to_bf16_bits(synth.normal(0, "embed", (vocab, shape["d_model"]), std=0.02))
    head = synth.f32_to_bf16_bits(synth.normal(0, "lm_head", (vocab, shape["d_model"]), std=0.02))
    fnorm = synth.f32_to_bf16_bits(synth.normal(0, "final_norm", (shape["d_model"],), std=0.1, mean=1.0))
    prompt = synth.uniform_int(0, "gen/8b_prompt", (B, S), vocab)
    toks, last, _ = _generate(lb, shape, layers, emb, head, fnorm, prompt, 0, n_new, L)
    _check_against_oracle(shape, layers, emb, head, fnorm, prompt, 0, toks, last, L, "bf16")


def test_generate_rejects_out_of_range_calls(lb):
    t = torch()
    shape = synth.SHAPES["tiny_f32"]
    vocab, L = 20, 8
    layers = [synth.block_weights(shape, layer=0)]
    wd = [{k: to_dev(v) for k, v in w.items()} for w in layers]
    emb = to_dev(synth.normal(0, "gen/e", (vocab, 64)))
    st, stk = lb.llama_stack_create(make_cfg(shape, L), 1, vocab, emb, [lb.make_weights(w) for w in wd],
                                    to_dev(np.ones(64, np.float32)), emb, 8)
    lb.check(st)
    try:
        kc = t.zeros((2, 2, L, 16), device="cuda")
        vc = t.zeros_like(kc)
        kvs = [lb.make_kv_cache(kc, vc, 2, L)]
        tok = t.zeros((2, 4), dtype=t.int32, device="cuda")
        out = t.zeros((2, 8), dtype=t.int32, device="cuda")
        logits = t.zeros((2, vocab), device="cuda")
        s = t.cuda.current_stream()
        assert lb.llama_stack_generate(stk, tok, 2, 4, 0, 5, kvs, out, logits, s) == lb.LLAMA_OK
        assert lb.llama_stack_generate(stk, tok, 2, 4, 0, 6, kvs, out, logits, s) == lb.LLAMA_ERR_RANGE
        assert lb.llama_stack_generate(stk, tok, 2, 4, 1, 5, kvs, out, logits, s) == lb.LLAMA_ERR_RANGE
        assert lb.llama_stack_generate(stk, tok, 2, 4, 0, 0, kvs, out, logits, s) == lb.LLAMA_ERR_INVALID_ARG
        assert lb.llama_stack_generate(stk, tok, 3, 4, 0, 2, kvs, out, logits, s) == lb.LLAMA_ERR_RANGE
        t.cuda.synchronize()
        assert lb.llama_stack_device_status(stk) == lb.LLAMA_OK
    finally:
        lb.llama_stack_destroy(stk)
