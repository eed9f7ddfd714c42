"""fp64 oracle of the Llama pre-norm decoder block (test infrastructure only).

Pages restated (cited by title and section):
  [EVT]  "The Evolving Transformer 04 · LLaMA" -- §00 Config, §01 Embeddings,
         §02 RoPE, §03 RMSNorm, §04 SwiGLU, §05 GQA, §06 Block, §07 Assemble.
  [L3B]  "Full Llama 3 transformer block" -- Overview, How it works, Watch-outs.
  [L4S]  "Llama 4 From Scratch" -- The idea, Worked example, In code.
  [ML2]  "Mini Llama 2 Implementation" -- RMS normalization, Rotary positional
         embeddings, Self-attention and transformer blocks.
  [G2L]  "From GPT-2 to Llama: four changes and the reason for each" --
         Positions become a rotation, The norm stops centring, The feed-forward
         grows a gate, Keys and values get shared, What the ML engineer watches.

Readings taken where the pages are open or disagree (each also listed in the
design notes):
  * RoPE pairs are interleaved (2i, 2i+1) ([EVT] §02, [ML2] Rotary), not the
    halves layout of [G2L]; frequency of pair i is theta^(-2i/D) ([ML2]
    Rotary, [L4S] Worked example); the position of query/key s is
    start_pos + s ([L3B] How it works: freqs_cis slice from start_pos).
  * RMSNorm adds eps to mean(x^2) inside the root ([EVT] §03, [L4S] In code,
    [ML2] RMS normalization, [G2L] The norm stops centring); no rounding.
  * Query head h reads KV head h // (H / G) ([EVT] §05 repeat_kv expands each
    KV head n_rep times in place); the cache stores K after RoPE and V as
    projected ([L3B] How it works: RoPE rotates Q and K, then keys/values are
    written into the cache).
  * Causal mask with cache offset: key j is visible to query i iff
    j <= start_pos + i ([L3B] How it works: mask shaped for the query length
    against the cached key length; [EVT] §05 tril mask is the start_pos = 0 case).
  * SwiGLU names follow [L3B]: W1 = gate, W3 = up, W2 = down; [EVT] §04 labels
    w2 up / w3 down -- the arithmetic is the same.

Parity pins (tests/test_oracle_pins.py) cover every function below; the whole
block has no printed worked example on the pages, so the block composition is
pinned through the special cases and invariants listed there (single-token
closed form, residual identity, pre-norm scale invariance, GQA == duplicated
MHA, causality, chunked prefill == one-shot == token-by-token decode).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "rms_norm", "rope_frequencies", "scale_rope_frequencies", "rope", "silu", "linear", "gqa_attention",
    "gqa_attention_rows", "block_forward", "block_forward_rows", "stack_forward", "greedy_generate",
    "swiglu", "moe_route", "moe_ffn", "block_residual_h",
    "ffn_hidden_dim", "kv_values_per_token", "block_param_count", "model_param_count",
]


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """u = x / sqrt(mean(x^2) + eps) * g over the last (model) axis.

    [EVT] §03 RMSNorm; [L3B] How it works (eps = norm_eps); [G2L] The norm stops
    centring (no mean subtraction, no shift).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope_frequencies(d_head: int, theta: float, scaling=None) -> np.ndarray:
    """Angular frequency of pair i: theta^(-2i / d_head), i = 0 .. d_head/2 - 1.

    [ML2] Rotary positional embeddings (theta ** (-2 * arange(D/2) / D));
    [L4S] Worked example; [EVT] §02 (base^(arange(0, D, 2) / D) inverted).
    With ``scaling`` (a dict, see :func:`scale_rope_frequencies`) the
    frequencies are stretched for contexts longer than the trained one.
    """
    i = np.arange(d_head // 2, dtype=np.float64)
    f = np.power(float(theta), -2.0 * i / d_head)
    return f if scaling is None else scale_rope_frequencies(f, scaling)


def scale_rope_frequencies(f: np.ndarray, scaling: dict) -> np.ndarray:
    """Llama 3.1 frequency stretch.  [G2L] Positions become a rotation: the
    slowest pairs are slowed by the factor, the fastest are left alone and the
    ones between are blended.

    scaling = {factor, low_freq_factor, high_freq_factor, original_max_pos}.
    A pair's wavelength is lam = 2 pi / f.  Pairs with lam shorter than
    original_max_pos / high_freq_factor keep f; pairs with lam longer than
    original_max_pos / low_freq_factor get f / factor; in between, f is blended
    linearly, (1 - w) f / factor + w f, with the weight
    w = (original_max_pos / lam - low_freq_factor) / (high_freq_factor - low_freq_factor),
    which is 1 at the short-wavelength edge and 0 at the long one.  The pages
    state the three bands, not the blend; the linear blend in turns-per-context
    is the reading taken (it is continuous at both edges).
    """
    f = np.asarray(f, dtype=np.float64)
    factor = float(scaling["factor"])
    lo, hi = float(scaling["low_freq_factor"]), float(scaling["high_freq_factor"])
    orig = float(scaling["original_max_pos"])
    lam = 2.0 * math.pi / f
    out = np.empty_like(f)
    for i, (fi, li) in enumerate(zip(f, lam)):
        if li < orig / hi:
            out[i] = fi
        elif li > orig / lo:
            out[i] = fi / factor
        else:
            w = (orig / li - lo) / (hi - lo)
            out[i] = (1.0 - w) * fi / factor + w * fi
    return out


def rope(x: np.ndarray, positions: np.ndarray, theta: float, layout: str = "interleaved",
         scaling=None) -> np.ndarray:
    """Rotate the pairs of x[..., S, heads, D] by p_s * f_i.

    (a, b) -> (a cos - b sin, a sin + b cos) with p_s = positions[s].
    layout "interleaved": pair i is (x[2i], x[2i+1]) -- [EVT] §02 RoPE
    (even/odd split, rotate, stack); [ML2] Rotary positional embeddings
    (reshape(-1, 2) real/imag form).  layout "halves": pair i is (x[i],
    x[i + D/2]) -- [G2L] Positions become a rotation (q cos + rotate_half(q)
    sin).  [L3B] How it works (positions start_pos .. start_pos + S - 1).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_frequencies(D, theta, scaling)[None, :]
    cos = np.cos(ang)[:, None, :]  # [S, 1, D/2] broadcast over heads
    sin = np.sin(ang)[:, None, :]
    if layout == "interleaved":
        ia, ib = slice(0, D, 2), slice(1, D, 2)
    elif layout == "halves":
        ia, ib = slice(0, D // 2), slice(D // 2, D)
    else:
        raise ValueError(f"unknown RoPE layout {layout!r}")
    a = x[..., ia]
    b = x[..., ib]
    out = np.empty_like(x)
    out[..., ia] = a * cos - b * sin
    out[..., ib] = a * sin + b * cos
    return out


def _rope_cfg(cfg, x, positions):
    return rope(x, positions, cfg["rope_theta"], cfg.get("rope_layout", "interleaved"), cfg.get("rope_scaling"))


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + e^-z).  [EVT] §04; [L4S] In code (Swish)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """nn.Linear without bias: y = x W^T with W stored [out, in].  [EVT] §05, §04."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def _softmax_rows(s: np.ndarray) -> np.ndarray:
    s = s - np.max(s, axis=-1, keepdims=True)
    p = np.exp(s)
    return p / np.sum(p, axis=-1, keepdims=True)


def gqa_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, start_pos: int) -> np.ndarray:
    """Causal grouped-query attention over the cache.

    q: [B, S, H, D] (already rotated); k_cache, v_cache: [B, G, L_max, D] holding
    keys/values of positions 0 .. start_pos + S - 1.  Query head h of token i
    attends to KV head h // (H / G) at key positions j <= start_pos + i with
    weights softmax_j(q . k_j / sqrt(D)); returns o [B, S, H, D].
    [EVT] §05 GQA (scores / sqrt(dk), -inf mask, softmax, @ value, repeat_kv);
    [L3B] How it works (cache read, offset mask).
    """
    B, S, H, D = q.shape
    G = k_cache.shape[1]
    r = H // G
    L = start_pos + S
    i = np.arange(S)[:, None]
    j = np.arange(L)[None, :]
    visible = j <= start_pos + i  # [S, L]
    o = np.empty((B, S, H, D), dtype=np.float64)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for h in range(H):
            g = h // r
            K = np.asarray(k_cache[b, g, :L], dtype=np.float64)
            V = np.asarray(v_cache[b, g, :L], dtype=np.float64)
            s = (np.asarray(q[b, :, h, :], dtype=np.float64) @ K.T) * scale
            s = np.where(visible, s, -np.inf)
            o[b, :, h, :] = _softmax_rows(s) @ V
    return o


def gqa_attention_rows(q_rows: np.ndarray, batch_idx, query_pos, k_cache, v_cache) -> np.ndarray:
    """Same attention for a list of single queries.

    q_rows: [n, H, D]; row n belongs to sequence batch_idx[n] and sits at absolute
    position query_pos[n], so it sees keys 0 .. query_pos[n].  Returns [n, H, D].
    """
    n, H, D = q_rows.shape
    G = k_cache.shape[1]
    r = H // G
    out = np.empty((n, H, D), dtype=np.float64)
    scale = 1.0 / math.sqrt(D)
    for t in range(n):
        b = int(batch_idx[t])
        L = int(query_pos[t]) + 1
        for h in range(H):
            g = h // r
            K = np.asarray(k_cache[b, g, :L], dtype=np.float64)
            V = np.asarray(v_cache[b, g, :L], dtype=np.float64)
            s = (K @ np.asarray(q_rows[t, h], dtype=np.float64)) * scale
            s = s - np.max(s)
            p = np.exp(s)
            out[t, h] = (p / np.sum(p)) @ V
    return out


def _dims(cfg):
    d = int(cfg["d_model"])
    H = int(cfg["n_heads"])
    G = int(cfg["n_kv_heads"])
    return d, H, G, d // H


def _project_qkv(cfg, w, x, start_pos):
    """attention_norm, Wq/Wk/Wv and RoPE on Q, K for all tokens of x [B, S, d]."""
    d, H, G, D = _dims(cfg)
    B, S, _ = x.shape
    u = rms_norm(x, w["attn_norm"], cfg["norm_eps"])
    q = linear(u, w["wq"]).reshape(B, S, H, D)
    k = linear(u, w["wk"]).reshape(B, S, G, D)
    v = linear(u, w["wv"]).reshape(B, S, G, D)
    pos = start_pos + np.arange(S)
    q = _rope_cfg(cfg, q, pos)
    k = _rope_cfg(cfg, k, pos)
    return q, k, v


def _write_cache(k_cache, v_cache, k, v, start_pos):
    """Store rotated K and V of positions start_pos .. start_pos + S - 1 ([L3B] How it works)."""
    S = k.shape[1]
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    kc[:, :, start_pos:start_pos + S, :] = k.transpose(0, 2, 1, 3)
    vc[:, :, start_pos:start_pos + S, :] = v.transpose(0, 2, 1, 3)
    return kc, vc


def swiglu(v: np.ndarray, w_gate, w_up, w_down) -> np.ndarray:
    """W2(SiLU(W1 v) * W3 v).  [EVT] §04 SwiGLU; [L3B] How it works."""
    return linear(silu(linear(v, w_gate)) * linear(v, w_up), w_down)


def moe_route(cfg: dict, w: dict, v: np.ndarray):
    """Router of a mixture-of-experts feed-forward: logits = v W_router^T over
    the n_experts experts; each token goes to the top_k largest logits (the
    lowest expert id among equal logits), weighted by a softmax over the
    logits of the chosen experts.  [G2L] The feed-forward grows a gate (a small
    layer that picks a few feed-forwards per token); [L4S] MoE (top-k of N
    experts, compute scales with k).  The pages name the top-k choice, not how
    the chosen outputs are weighted: a softmax over the chosen logits is the
    reading taken.
    Returns (ids int [T, k], weights [T, k], logits [T, E]) for v [T, d].
    """
    k = int(cfg["top_k"])
    logits = linear(v, w["router"])
    ids = np.argsort(-logits, axis=-1, kind="stable")[:, :k]  # stable: equal logits keep id order
    top = np.take_along_axis(logits, ids, -1)
    e = np.exp(top - top.max(-1, keepdims=True))
    return ids, e / e.sum(-1, keepdims=True), logits


def moe_ffn(cfg: dict, w: dict, v: np.ndarray, route=None) -> np.ndarray:
    """Mixture-of-experts SwiGLU feed-forward on normalised tokens v [..., d]:
    sum over the k chosen experts of weight * expert_e(v), plus the always-on
    shared expert when the block has one.  [L4S] MoE with a shared expert
    (Llama 4 keeps one shared expert every token uses).  Experts are stacked:
    w_gate, w_up [E, F, d], w_down [E, d, F]; shared_gate, shared_up [F_s, d],
    shared_down [d, F_s].  route = (ids, weights) overrides the router's
    choice (used to evaluate the block on another implementation's routing).
    """
    shp = v.shape
    v = np.asarray(v, dtype=np.float64).reshape(-1, shp[-1])
    ids, wts = route if route is not None else moe_route(cfg, w, v)[:2]
    out = np.zeros_like(v)
    for e in np.unique(ids):
        rows, slot = np.nonzero(ids == e)
        ye = swiglu(v[rows], w["w_gate"][e], w["w_up"][e], w["w_down"][e])
        np.add.at(out, rows, wts[rows, slot][:, None] * ye)
    if cfg.get("d_ff_shared", 0):
        out = out + swiglu(v, w["shared_gate"], w["shared_up"], w["shared_down"])
    return out.reshape(shp)


def _ffn(cfg, w, h, route=None):
    """ffn_norm then the feed-forward: SwiGLU W2(SiLU(W1 v) * W3 v) ([L3B] How
    it works; [EVT] §04), or the mixture of experts when cfg has n_experts."""
    v2 = rms_norm(h, w["ffn_norm"], cfg["norm_eps"])
    if cfg.get("n_experts", 0):
        return moe_ffn(cfg, w, v2, route)
    return swiglu(v2, w["w_gate"], w["w_up"], w["w_down"])


def block_forward(cfg: dict, w: dict, x: np.ndarray, start_pos: int, k_cache: np.ndarray,
                  v_cache: np.ndarray, route=None):
    """One pre-norm block: h = x + Attn(RMSNorm(x)); y = h + FFN(RMSNorm(h)).

    x: [B, S, d]; caches [B_max, G, L_max, D] (B_max >= B; rows >= B untouched).
    Returns (y, k_cache', v_cache') -- the caches are new fp64 arrays with
    positions start_pos .. start_pos + S - 1 of sequences 0 .. B - 1 written.
    [L3B] Overview / How it works (the two residual branches, untied norms);
    [EVT] §06 Block; [ML2] Self-attention and transformer blocks.
    route: for a mixture-of-experts block, optional (ids, weights) [B*S, k]
    replacing the router's choice (see moe_ffn).
    """
    x = np.asarray(x, dtype=np.float64)
    B = x.shape[0]
    h, kc, vc = block_residual_h(cfg, w, x, start_pos, k_cache, v_cache)
    y = h + _ffn(cfg, w, h, route)
    kfull = np.array(k_cache, dtype=np.float64, copy=True)
    vfull = np.array(v_cache, dtype=np.float64, copy=True)
    kfull[:B] = kc
    vfull[:B] = vc
    return y, kfull, vfull


def block_residual_h(cfg: dict, w: dict, x: np.ndarray, start_pos: int, k_cache, v_cache):
    """The attention half of the block: h = x + Wo Attn(RMSNorm(x)), plus the
    caches of sequences 0 .. B - 1 with the new keys/values written.  The
    first residual branch of [L3B] How it works; :func:`block_forward` adds the
    feed-forward branch to it."""
    d, H, G, D = _dims(cfg)
    x = np.asarray(x, dtype=np.float64)
    B, S, _ = x.shape
    q, k, v = _project_qkv(cfg, w, x, start_pos)
    kc, vc = _write_cache(np.asarray(k_cache, dtype=np.float64)[:B], np.asarray(v_cache, dtype=np.float64)[:B],
                          k, v, start_pos)
    o = gqa_attention(q, kc, vc, start_pos).reshape(B, S, H * D)
    return x + linear(o, w["wo"]), kc, vc


def block_forward_rows(cfg: dict, w: dict, x: np.ndarray, start_pos: int, k_cache, v_cache, rows):
    """The block output y at selected (b, s) rows only, plus the written K/V slice.

    Every key/value of positions < start_pos + S is still computed (all queries
    may see them); queries, the O projection and the FFN run only for the
    selected rows.  Same definition as :func:`block_forward`, restricted.
    Returns (y_rows [n, d], k_new [B, G, S, D], v_new [B, G, S, D]).
    """
    d, H, G, D = _dims(cfg)
    x = np.asarray(x, dtype=np.float64)
    B, S, _ = x.shape
    u = rms_norm(x, w["attn_norm"], cfg["norm_eps"])
    pos = start_pos + np.arange(S)
    k = _rope_cfg(cfg, linear(u, w["wk"]).reshape(B, S, G, D), pos)
    v = linear(u, w["wv"]).reshape(B, S, G, D)
    kc, vc = _write_cache(np.asarray(k_cache[:B], dtype=np.float64), np.asarray(v_cache[:B], dtype=np.float64),
                          k, v, start_pos)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    bi, si = rows[:, 0], rows[:, 1]
    ur = u[bi, si]  # [n, d]
    qr = linear(ur, w["wq"]).reshape(-1, 1, H, D)
    qr = np.stack([_rope_cfg(cfg, qr[t:t + 1], np.array([start_pos + si[t]]))[0, 0]
                   for t in range(len(si))]) if len(si) else qr.reshape(0, H, D)
    o = gqa_attention_rows(qr, bi, start_pos + si, kc, vc).reshape(-1, H * D)
    h = x[bi, si] + linear(o, w["wo"])
    y = h + _ffn(cfg, w, h)
    k_new = kc[:, :, start_pos:start_pos + S, :]
    v_new = vc[:, :, start_pos:start_pos + S, :]
    return y, k_new, v_new


def stack_forward(cfg: dict, layers, embed, final_norm, lm_head, tokens, start_pos: int, caches):
    """Token embedding -> N blocks -> final RMSNorm -> untied LM head (logits).

    tokens: int [B, S]; layers: list of weight dicts; caches: list of (k, v).
    [EVT] §01 Embeddings (wte only, no position table), §07 Assemble (blocks,
    final norm, lm_head); untied per [EVT] §00 (~8.0B with untied embeddings).
    Returns (logits [B, S, vocab], new caches).
    """
    x = np.asarray(embed, dtype=np.float64)[np.asarray(tokens)]
    new_caches = []
    for w, (kc, vc) in zip(layers, caches):
        x, kc2, vc2 = block_forward(cfg, w, x, start_pos, kc, vc)
        new_caches.append((kc2, vc2))
    n = rms_norm(x, final_norm, cfg["norm_eps"])
    return linear(n, lm_head), new_caches


def greedy_generate(cfg: dict, layers, embed, final_norm, lm_head, prompt, start_pos: int, caches, n_new: int):
    """Greedy decoding through the stack with the KV cache.

    The prompt (int [B, S]) runs through the stack at start_pos, filling every
    layer's cache; the next token of each sequence is the arg-max of the logits
    at its last prompt position (the lowest id among equal maxima); that token
    is then run as a one-token step at the next position, and so on, n_new
    tokens in all.  [L3B] How it works (the cache-backed forward at start_pos,
    one new token per step once the prompt is cached); [EVT] §07 Assemble
    (logits of the last position choose the next token).
    Returns (tokens [B, n_new], logits [B, vocab] of the last step, caches).
    """
    prompt = np.asarray(prompt)
    B, S = prompt.shape
    out = np.zeros((B, n_new), dtype=np.int64)
    logits, caches = stack_forward(cfg, layers, embed, final_norm, lm_head, prompt, start_pos, caches)
    last = logits[:, -1]
    pos = start_pos + S
    for i in range(n_new):
        out[:, i] = np.argmax(last, axis=-1)  # first index of the maximum
        if i + 1 == n_new:
            break
        logits, caches = stack_forward(cfg, layers, embed, final_norm, lm_head, out[:, i:i + 1], pos, caches)
        last = logits[:, -1]
        pos += 1
    return out, last, caches


# ---------------------------------------------------------------------------
# Shape arithmetic the pages fix.
# ---------------------------------------------------------------------------

def ffn_hidden_dim(d_model: int, multiple_of: int, ffn_dim_multiplier=None) -> int:
    """SwiGLU inner width: 4d, then 2/3 (floor), then x multiplier (floor), then
    round up to a multiple of multiple_of.  [L3B] How it works (FeedForward
    constructor: hidden_dim = 4 * dim, 2/3 shrink, optional ffn_dim_multiplier,
    multiple_of rounding); [G2L] The feed-forward grows a gate (f = 8d/3)."""
    h = 4 * d_model
    h = int(2 * h / 3)
    if ffn_dim_multiplier is not None:
        h = int(ffn_dim_multiplier * h)
    return multiple_of * ((h + multiple_of - 1) // multiple_of)


def kv_values_per_token(n_layers: int, n_kv_heads: int, d_head: int) -> int:
    """Cached numbers per token: 2 (K and V) x layers x KV heads x head width.
    [L4S] Worked example; [G2L] What the ML engineer watches."""
    return 2 * n_layers * n_kv_heads * d_head


def block_param_count(d_model: int, n_heads: int, n_kv_heads: int, d_ff: int, norms: bool = True) -> dict:
    """Parameter counts of one block (no biases): attention, FFN, norms, total."""
    D = d_model // n_heads
    attn = d_model * n_heads * D + 2 * d_model * n_kv_heads * D + n_heads * D * d_model
    ffn = 3 * d_model * d_ff
    nrm = 2 * d_model if norms else 0
    return {"attention": attn, "ffn": ffn, "norms": nrm, "total": attn + ffn + nrm}


def model_param_count(d_model, n_heads, n_kv_heads, d_ff, n_layers, vocab, tied: bool) -> int:
    """Embedding + N blocks + final norm (+ LM head when untied).  [EVT] §07; §00."""
    blk = block_param_count(d_model, n_heads, n_kv_heads, d_ff)["total"]
    emb = vocab * d_model
    return n_layers * blk + emb + d_model + (0 if tied else emb)
