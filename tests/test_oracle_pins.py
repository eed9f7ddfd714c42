"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages print, a closed form,
an invariant the mathematics fixes, or a brute-force restatement, chosen so
that a plausible slip (dropped term, wrong sign or index, transposed operand,
wrong grouping or exponent) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))

TINY = dict(d_model=64, n_heads=4, n_kv_heads=2, d_ff=192, norm_eps=1e-5, rope_theta=1e4)


def _rng(tag, shape, std=1.0, mean=0.0):
    return synth.normal(0, "pins/" + tag, shape, std=std, mean=mean).astype(np.float64)


def _tiny_weights(cfg, seed_tag="w"):
    shp = synth.weight_shapes(**cfg)
    w = {}
    for n, s in shp.items():
        if n.endswith("norm"):
            w[n] = _rng(seed_tag + n, s, std=0.1, mean=1.0)
        else:
            w[n] = _rng(seed_tag + n, s, std=0.2)  # larger than 0.02 so every branch matters
    return w


# ---------------------------------------------------------------- RoPE -------

def test_rope_periods_match_printed_values():
    g = GOLDEN["rope_periods_smollm2"]
    f = oracle.rope_frequencies(g["d_head"], g["theta"])
    periods = 2 * math.pi / f
    assert abs(periods.min() - g["fastest_period_positions"]) <= g["fastest_tolerance"]
    assert abs(periods.max() - g["slowest_period_positions"]) <= g["slowest_tolerance"]
    assert len(f) == g["d_head"] // 2
    assert np.all(np.diff(f) < 0)  # pair 0 fastest


def test_rope_score_depends_only_on_offset():
    g = GOLDEN["rope_relative_score_smollm2"]
    D, theta = 64, 1e5
    q = _rng("rope_q", (1, 1, D))
    k = _rng("rope_k", (1, 1, D))

    def score(m, n):
        qm = oracle.rope(q, np.array([m]), theta)
        kn = oracle.rope(k, np.array([n]), theta)
        return float(np.sum(qm * kn))

    (m1, n1), (m2, n2) = g["pairs_equal"]
    s1, s2 = score(m1, n1), score(m2, n2)
    s3 = score(*g["pair_different"])
    assert abs(s1 - s2) <= 1e-12 * max(1.0, abs(s1))
    assert abs(s1 - s3) > 1e-3


def test_rope_identity_at_position_zero_and_norm_preserving():
    x = _rng("rope_x", (3, 5, 16))
    y0 = oracle.rope(x, np.zeros(3), 1e4)
    assert np.array_equal(y0, x)
    y = oracle.rope(x, np.array([1.0, 77.0, 4095.0]), 5e5)
    n_in = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_out = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13, atol=1e-13)


def test_rope_unit_vector_closed_form():
    # pair 0 has frequency 1: (1, 0) at position p becomes (cos p, sin p);
    # (0, 1) becomes (-sin p, cos p) -- fixes the sign convention of the rotation.
    D = 8
    x = np.zeros((1, 2, D))
    x[0, 0, 0] = 1.0
    x[0, 1, 1] = 1.0
    p = 3.0
    y = oracle.rope(x, np.array([p]), 1e4)
    assert y[0, 0, 0] == pytest.approx(math.cos(p), abs=1e-15)
    assert y[0, 0, 1] == pytest.approx(math.sin(p), abs=1e-15)
    assert y[0, 1, 0] == pytest.approx(-math.sin(p), abs=1e-15)
    assert y[0, 1, 1] == pytest.approx(math.cos(p), abs=1e-15)
    # pair 1 turns at theta^(-2/D)
    x2 = np.zeros((1, 1, D))
    x2[0, 0, 2] = 1.0
    y2 = oracle.rope(x2, np.array([p]), 1e4)
    a = p * 1e4 ** (-2.0 / D)
    assert y2[0, 0, 2] == pytest.approx(math.cos(a), abs=1e-15)
    assert y2[0, 0, 3] == pytest.approx(math.sin(a), abs=1e-15)


def test_rope_equals_complex_multiplication_on_interleaved_pairs():
    # The complex form: (x[2i] + j x[2i+1]) * exp(j p f_i), pairs read with reshape(-1, 2).
    D, theta = 16, 5e5
    x = _rng("rope_c", (4, 2, D))
    pos = np.array([0.0, 5.0, 1234.0, 8191.0])
    z = x.reshape(4, 2, D // 2, 2)
    zc = z[..., 0] + 1j * z[..., 1]
    f = theta ** (-np.arange(0, D, 2) / D)
    rot = np.exp(1j * pos[:, None, None] * f[None, None, :])
    w = zc * rot
    ref = np.stack([w.real, w.imag], axis=-1).reshape(4, 2, D)
    np.testing.assert_allclose(oracle.rope(x, pos, theta), ref, rtol=0, atol=1e-12)
    # the halves layout (pairs i, i + D/2) is a different map: must not match
    a, b = x[..., : D // 2], x[..., D // 2:]
    ang = pos[:, None, None] * f[None, None, :]
    halves = np.concatenate([a * np.cos(ang) - b * np.sin(ang), a * np.sin(ang) + b * np.cos(ang)], -1)
    assert np.max(np.abs(halves - oracle.rope(x, pos, theta))) > 1e-2


def _halves_to_interleaved(D):
    """Index map: interleaved position 2i <- halves position i, 2i+1 <- i + D/2."""
    idx = np.empty(D, dtype=np.int64)
    idx[0::2] = np.arange(D // 2)
    idx[1::2] = np.arange(D // 2) + D // 2
    return idx


def test_rope_halves_equals_complex_multiplication_on_halves():
    # the halves form: (x[i] + j x[i + D/2]) * exp(j p f_i)
    D, theta = 16, 1e5
    x = _rng("rope_h", (3, 2, D))
    pos = np.array([0.0, 9.0, 3000.0])
    zc = x[..., : D // 2] + 1j * x[..., D // 2:]
    f = theta ** (-np.arange(0, D, 2) / D)
    w = zc * np.exp(1j * pos[:, None, None] * f[None, None, :])
    ref = np.concatenate([w.real, w.imag], -1)
    np.testing.assert_allclose(oracle.rope(x, pos, theta, layout="halves"), ref, rtol=0, atol=1e-12)


def test_rope_halves_is_interleaved_rope_of_the_permuted_vector():
    # Reordering each head as (x0, x_{D/2}, x1, x_{D/2+1}, ...) turns the halves rotation into the
    # interleaved one; dot products are unchanged by a common reordering of q and k.
    D, theta = 32, 5e5
    x = _rng("rope_p", (4, 3, D))
    pos = np.array([1.0, 17.0, 4095.0, 20000.0])
    idx = _halves_to_interleaved(D)
    via_interleaved = np.empty_like(x)
    via_interleaved[..., idx] = oracle.rope(x[..., idx], pos, theta)
    np.testing.assert_allclose(oracle.rope(x, pos, theta, layout="halves"), via_interleaved, rtol=0, atol=1e-12)


def test_rope_halves_score_depends_only_on_offset_and_keeps_norms():
    D, theta = 64, 1e5
    q = _rng("rope_hq", (1, 1, D))
    k = _rng("rope_hk", (1, 1, D))

    def score(m, n):
        return float(np.sum(oracle.rope(q, np.array([m]), theta, "halves") *
                            oracle.rope(k, np.array([n]), theta, "halves")))

    assert abs(score(10, 3) - score(1010, 1003)) <= 1e-12 * abs(score(10, 3))
    assert abs(score(10, 3) - score(10, 4)) > 1e-3
    y = oracle.rope(q, np.array([321.0]), theta, "halves")
    np.testing.assert_allclose(np.linalg.norm(y), np.linalg.norm(q), rtol=1e-13)


LLAMA31_SCALING = dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)


def test_rope_scaling_bands_match_printed_counts():
    g = GOLDEN["rope_scaling_llama31_8b"]
    f = oracle.rope_frequencies(g["d_head"], g["theta"])
    fs = oracle.rope_frequencies(g["d_head"], g["theta"], LLAMA31_SCALING)
    assert len(f) == g["pairs"]
    ratio = f / fs
    unchanged = int(np.sum(np.abs(ratio - 1.0) < 1e-12))
    slowed = int(np.sum(np.abs(ratio - g["slow_factor"]) < 1e-9))
    blended = int(np.sum((ratio > 1.0 + 1e-12) & (ratio < g["slow_factor"] - 1e-9)))
    assert (unchanged, slowed, blended) == (g["unchanged"], g["slowed"], g["blended"])
    # the fastest pairs are the unchanged ones, the slowest the slowed ones
    assert np.all(np.abs(ratio[: g["unchanged"]] - 1.0) < 1e-12)
    assert np.all(np.abs(ratio[-g["slowed"]:] - g["slow_factor"]) < 1e-9)
    assert g["max_pos"] // g["original_max_pos"] == 16  # 8192 -> 131072 positions


def test_rope_scaling_is_continuous_and_monotone():
    orig, lo, hi, fac = 8192.0, 1.0, 4.0, 8.0
    sc = dict(factor=fac, low_freq_factor=lo, high_freq_factor=hi, original_max_pos=orig)
    eps = 1e-9
    for lam in (orig / hi, orig / lo):  # the two band edges
        f_in, f_out = 2 * math.pi / (lam * (1 - eps)), 2 * math.pi / (lam * (1 + eps))
        a, b = oracle.scale_rope_frequencies(np.array([f_in, f_out]), sc)
        assert abs(a - b) <= 1e-6 * a
    lam = np.linspace(100.0, 3 * orig, 2001)
    fs = oracle.scale_rope_frequencies(2 * math.pi / lam, sc)
    assert np.all(np.diff(fs) < 0)  # longer wavelength, lower scaled frequency
    # factor 1 is the identity
    f = oracle.rope_frequencies(128, 5e5)
    np.testing.assert_allclose(oracle.scale_rope_frequencies(f, dict(sc, factor=1.0)), f, rtol=1e-15, atol=0)


def test_rope_with_scaling_rotates_by_the_scaled_frequencies():
    D, theta = 128, 5e5
    x = np.zeros((1, 1, D))
    x[0, 0, 2 * 63] = 1.0  # the slowest pair
    p = 100000.0
    y = oracle.rope(x, np.array([p]), theta, scaling=LLAMA31_SCALING)
    a = p * theta ** (-126.0 / D) / 8.0
    assert y[0, 0, 126] == pytest.approx(math.cos(a), abs=1e-12)
    assert y[0, 0, 127] == pytest.approx(math.sin(a), abs=1e-12)


# ------------------------------------------------------------- RMSNorm -------

def test_rmsnorm_unit_gain_gives_unit_rms():
    x = _rng("rms_x", (7, 576), std=3.0)
    eps = 1e-5
    u = oracle.rms_norm(x, np.ones(576), eps)
    ms = np.mean(x * x, axis=-1)
    rms_out = np.sqrt(np.mean(u * u, axis=-1))
    np.testing.assert_allclose(rms_out, np.sqrt(ms / (ms + eps)), rtol=1e-13)
    np.testing.assert_allclose(rms_out, 1.0, atol=1e-5)


def test_rmsnorm_closed_forms_and_no_centring():
    g = np.array([1.0, 2.0, 3.0, 4.0])
    assert np.array_equal(oracle.rms_norm(np.ones(4), g, 0.0), g)
    np.testing.assert_allclose(oracle.rms_norm(np.array([2.0, -2.0, 2.0, -2.0]), np.ones(4), 0.0),
                               [1.0, -1.0, 1.0, -1.0], rtol=0, atol=1e-15)
    # a constant offset is not removed (no mean subtraction): [5, 5, 5, 5] -> [1, 1, 1, 1]
    np.testing.assert_allclose(oracle.rms_norm(np.full(4, 5.0), np.ones(4), 0.0), np.ones(4), atol=1e-15)
    # eps sits inside the root: x = [1, 1], eps = 3 -> 1 / sqrt(1 + 3) = 0.5
    np.testing.assert_allclose(oracle.rms_norm(np.ones(2), np.ones(2), 3.0), [0.5, 0.5], atol=1e-15)


def test_rmsnorm_scale_invariance():
    x = _rng("rms_s", (3, 64))
    g = _rng("rms_g", (64,), std=0.1, mean=1.0)
    np.testing.assert_allclose(oracle.rms_norm(17.0 * x, g, 0.0), oracle.rms_norm(x, g, 0.0), rtol=1e-13)


# ------------------------------------------------------------- SwiGLU --------

def test_silu_closed_forms():
    assert oracle.silu(np.array(0.0)) == 0.0
    assert float(oracle.silu(np.array(1.0))) == pytest.approx(0.7310585786300049, abs=1e-15)  # sigmoid(1)
    assert float(oracle.silu(np.array(-1.0))) == pytest.approx(-0.2689414213699951, abs=1e-15)
    assert float(oracle.silu(np.array(30.0))) == pytest.approx(30.0, abs=1e-10)
    assert abs(float(oracle.silu(np.array(-30.0)))) < 1e-11


def test_swiglu_gate_times_up_elementwise():
    # identity gate / up / down of width d: FFN(v) = SiLU(v) * v elementwise
    d = 8
    cfg = dict(TINY, d_model=d, n_heads=2, n_kv_heads=1, d_ff=d, norm_eps=0.0)
    w = {"ffn_norm": np.ones(d), "w_gate": np.eye(d), "w_up": np.eye(d), "w_down": np.eye(d)}
    h = np.array([[[2.0, -2.0, 2.0, -2.0, 2.0, -2.0, 2.0, -2.0]]])  # RMS 2 -> normalised to +-1
    out = oracle.llama_block._ffn(cfg, w, h)
    s1 = 0.7310585786300049  # sigmoid(1)
    # v = +1: SiLU(1) * 1 = sigmoid(1); v = -1: SiLU(-1) * (-1) = sigmoid(-1) = 1 - sigmoid(1)
    np.testing.assert_allclose(out[0, 0], np.tile([s1, 1.0 - s1], 4), atol=1e-14)


def test_swiglu_gate_and_up_are_not_interchangeable():
    d = 4
    cfg = dict(TINY, d_model=d, n_heads=2, n_kv_heads=1, d_ff=d, norm_eps=0.0)
    h = np.array([[[1.0, -1.0, 1.0, -1.0]]])
    up_scaled = {"ffn_norm": np.ones(d), "w_gate": np.eye(d), "w_up": 2.0 * np.eye(d), "w_down": np.eye(d)}
    gate_scaled = {"ffn_norm": np.ones(d), "w_gate": 2.0 * np.eye(d), "w_up": np.eye(d), "w_down": np.eye(d)}
    a = oracle.llama_block._ffn(cfg, up_scaled, h)[0, 0]
    b = oracle.llama_block._ffn(cfg, gate_scaled, h)[0, 0]
    s1 = 0.7310585786300049
    np.testing.assert_allclose(a[0], 2.0 * s1, atol=1e-14)  # SiLU(1) * 2
    np.testing.assert_allclose(b[0], 2.0 / (1.0 + math.exp(-2.0)), atol=1e-14)  # SiLU(2) * 1


def test_ffn_width_rule_matches_printed_widths():
    for c in GOLDEN["ffn_widths"]["cases"]:
        assert oracle.ffn_hidden_dim(c["d_model"], c["multiple_of"], c["ffn_dim_multiplier"]) == c["hidden"]
    # 3 d f = 8 d^2 at f = 8d/3 (parameter parity with a 4d two-matrix MLP)
    assert 3 * 576 * 1536 == 8 * 576 * 576


# ---------------------------------------------------------- attention --------

def _brute_attention(q, kc, vc, start_pos):
    """Scalar loops with math.exp: materialised per-head K/V copy (repeat_kv),
    explicit lower-triangular visibility, full softmax row."""
    B, S, H, D = q.shape
    G = kc.shape[1]
    r = H // G
    out = np.zeros_like(q)
    for b in range(B):
        kr = [kc[b, hh // r] for hh in range(H)]  # repeat_kv copy
        vr = [vc[b, hh // r] for hh in range(H)]
        for h in range(H):
            for i in range(S):
                scores = []
                for j in range(start_pos + S):
                    if j <= start_pos + i:
                        scores.append(sum(q[b, i, h, t] * kr[h][j, t] for t in range(D)) / math.sqrt(D))
                m = max(scores)
                e = [math.exp(s - m) for s in scores]
                z = sum(e)
                for t in range(D):
                    out[b, i, h, t] = sum(e[j] / z * vr[h][j, t] for j in range(len(e)))
    return out


@pytest.mark.parametrize("H,G,start_pos", [(4, 2, 0), (4, 4, 0), (6, 2, 3), (3, 1, 2)])
def test_attention_matches_bruteforce(H, G, start_pos):
    B, S, D = 2, 5, 4
    q = _rng(f"att_q{H}{G}", (B, S, H, D))
    kc = _rng(f"att_k{H}{G}", (B, G, start_pos + S + 2, D))
    vc = _rng(f"att_v{H}{G}", (B, G, start_pos + S + 2, D))
    ref = _brute_attention(q, kc, vc, start_pos)
    np.testing.assert_allclose(oracle.gqa_attention(q, kc, vc, start_pos), ref, rtol=0, atol=1e-12)
    rows = [(0, 0), (1, 4), (0, 2)]
    qr = np.stack([q[b, s] for b, s in rows])
    got = oracle.gqa_attention_rows(qr, [b for b, _ in rows], [start_pos + s for _, s in rows], kc, vc)
    np.testing.assert_allclose(got, np.stack([ref[b, s] for b, s in rows]), rtol=0, atol=1e-12)


def test_attention_first_query_sees_only_itself():
    q = _rng("att1_q", (1, 3, 2, 4))
    kc = _rng("att1_k", (1, 1, 3, 4))
    vc = _rng("att1_v", (1, 1, 3, 4))
    o = oracle.gqa_attention(q, kc, vc, 0)
    np.testing.assert_array_equal(o[0, 0, 0], vc[0, 0, 0])
    np.testing.assert_array_equal(o[0, 0, 1], vc[0, 0, 0])


def test_attention_equal_scores_average_values():
    # all keys equal -> uniform weights -> mean of visible values
    q = _rng("att2_q", (1, 4, 1, 4))
    kc = np.tile(_rng("att2_k", (1, 1, 1, 4)), (1, 1, 4, 1))
    vc = _rng("att2_v", (1, 1, 4, 4))
    o = oracle.gqa_attention(q, kc, vc, 0)
    for i in range(4):
        np.testing.assert_allclose(o[0, i, 0], vc[0, 0, : i + 1].mean(axis=0), atol=1e-14)


# --------------------------------------------------------------- block -------

def _tiny_inputs(cfg, B=1, S=6, Lmax=12, tag="blk"):
    w = _tiny_weights(cfg, tag)
    x = _rng(tag + "x", (B, S, cfg["d_model"]))
    G, D = cfg["n_kv_heads"], cfg["d_model"] // cfg["n_heads"]
    kc = np.zeros((B, G, Lmax, D))
    vc = np.zeros((B, G, Lmax, D))
    return w, x, kc, vc


def test_block_single_token_closed_form():
    # S = 1 at start_pos 0: the only visible key is the token itself, so every
    # query head h outputs v of KV head h // r, whatever q, k and RoPE are.
    cfg = TINY
    d, H, G = 64, 4, 2
    D, r = d // H, H // G
    w, x, kc, vc = _tiny_inputs(cfg, B=2, S=1, Lmax=4, tag="st")
    y, kc2, vc2 = oracle.block_forward(cfg, w, x, 0, kc, vc)
    eps = cfg["norm_eps"]
    for b in range(2):
        xt = x[b, 0]
        u = xt / math.sqrt(float(np.mean(xt ** 2)) + eps) * w["attn_norm"]
        v = w["wv"] @ u
        o = np.concatenate([v[(h // r) * D:(h // r + 1) * D] for h in range(H)])
        h1 = xt + w["wo"] @ o
        v2 = h1 / math.sqrt(float(np.mean(h1 ** 2)) + eps) * w["ffn_norm"]
        gte = w["w_gate"] @ v2
        a = gte / (1 + np.exp(-gte)) * (w["w_up"] @ v2)
        np.testing.assert_allclose(y[b, 0], h1 + w["w_down"] @ a, rtol=0, atol=1e-12)
        # position 0: RoPE is the identity, so the cached key is the raw projection
        np.testing.assert_allclose(kc2[b, :, 0].reshape(-1), w["wk"] @ u, atol=1e-13)
        np.testing.assert_allclose(vc2[b, :, 0].reshape(-1), v, atol=1e-13)


def test_block_residual_identity_when_output_projections_vanish():
    cfg = TINY
    w, x, kc, vc = _tiny_inputs(cfg, tag="ri")
    w["wo"] = np.zeros_like(w["wo"])
    w["w_down"] = np.zeros_like(w["w_down"])
    y, kc2, _ = oracle.block_forward(cfg, w, x, 0, kc, vc)
    np.testing.assert_array_equal(y, x)
    assert np.any(kc2[:, :, :6] != 0) and np.all(kc2[:, :, 6:] == 0)


def test_block_is_pre_norm_attention_branch_scale_invariant():
    cfg = dict(TINY, norm_eps=0.0)
    w, x, kc, vc = _tiny_inputs(cfg, tag="pn")
    w["w_down"] = np.zeros_like(w["w_down"])
    y1, _, _ = oracle.block_forward(cfg, w, x, 0, kc, vc)
    y2, _, _ = oracle.block_forward(cfg, w, 9.0 * x, 0, kc, vc)
    np.testing.assert_allclose(y2 - 9.0 * x, y1 - x, rtol=1e-11, atol=1e-12)


def test_block_identical_tokens_attention_output_is_v():
    # all rows of x equal -> all values equal -> attention returns v for every
    # row whatever the (RoPE-dependent) weights are: softmax rows sum to one.
    cfg = TINY
    w, _, kc, vc = _tiny_inputs(cfg, tag="it")
    x = np.tile(_rng("it_row", (1, 1, 64)), (1, 6, 1))
    w["w_down"] = np.zeros_like(w["w_down"])
    y, _, _ = oracle.block_forward(cfg, w, x, 0, kc, vc)
    y1, _, _ = oracle.block_forward(cfg, w, x[:, :1], 0, kc, vc)
    for i in range(6):
        np.testing.assert_allclose(y[0, i], y1[0, 0], atol=1e-12)


def test_gqa_equals_mha_with_duplicated_kv_heads_and_tiling_differs():
    cfg = dict(TINY, n_heads=4, n_kv_heads=2)
    w, x, kc, vc = _tiny_inputs(cfg, tag="gq")
    H, G, D = 4, 2, 16
    r = H // G
    y_gqa, _, _ = oracle.block_forward(cfg, w, x, 0, kc, vc)

    def expand(wkv, order):
        return np.concatenate([wkv[order(h) * D:(order(h) + 1) * D] for h in range(H)])

    mha = dict(cfg, n_kv_heads=H)
    kc4 = np.zeros((1, H, 12, D))
    w_int = dict(w, wk=expand(w["wk"], lambda h: h // r), wv=expand(w["wv"], lambda h: h // r))
    y_mha, _, _ = oracle.block_forward(mha, w_int, x, 0, kc4, kc4)
    np.testing.assert_allclose(y_mha, y_gqa, rtol=0, atol=1e-13)
    w_tile = dict(w, wk=expand(w["wk"], lambda h: h % G), wv=expand(w["wv"], lambda h: h % G))
    y_tile, _, _ = oracle.block_forward(mha, w_tile, x, 0, kc4, kc4)
    assert np.max(np.abs(y_tile - y_gqa)) > 1e-3


def test_block_causality():
    cfg = TINY
    w, x, kc, vc = _tiny_inputs(cfg, tag="ca")
    y, _, _ = oracle.block_forward(cfg, w, x, 0, kc, vc)
    x2 = x.copy()
    x2[:, 4:] += 5.0
    y2, _, _ = oracle.block_forward(cfg, w, x2, 0, kc, vc)
    np.testing.assert_allclose(y2[:, :4], y[:, :4], rtol=0, atol=1e-13)
    assert np.max(np.abs(y2[:, 4:] - y[:, 4:])) > 1e-2


def test_chunked_prefill_equals_oneshot_equals_token_by_token():
    cfg = TINY
    B, S, L = 2, 7, 10
    w, x, kc, vc = _tiny_inputs(cfg, B=B, S=S, Lmax=L, tag="ch")
    y_one, k_one, v_one = oracle.block_forward(cfg, w, x, 0, kc, vc)
    ya, k1, v1 = oracle.block_forward(cfg, w, x[:, :3], 0, kc, vc)
    yb, k2, v2 = oracle.block_forward(cfg, w, x[:, 3:], 3, k1, v1)
    np.testing.assert_allclose(np.concatenate([ya, yb], 1), y_one, rtol=0, atol=1e-12)
    np.testing.assert_allclose(k2, k_one, atol=1e-13)
    kt, vt = kc, vc
    ys = []
    for s in range(S):
        yt, kt, vt = oracle.block_forward(cfg, w, x[:, s:s + 1], s, kt, vt)
        ys.append(yt)
    np.testing.assert_allclose(np.concatenate(ys, 1), y_one, rtol=0, atol=1e-12)
    np.testing.assert_allclose(vt, v_one, atol=1e-13)
    assert np.all(k_one[:, :, S:] == 0)


def test_block_forward_rows_matches_full_block():
    cfg = dict(TINY, n_heads=4, n_kv_heads=1)
    w, x, kc, vc = _tiny_inputs(cfg, B=2, S=6, Lmax=9, tag="rw")
    kc[:, :, :2] = _rng("rw_kc", (2, 1, 2, 16))
    vc[:, :, :2] = _rng("rw_vc", (2, 1, 2, 16))
    y, kfull, vfull = oracle.block_forward(cfg, w, x[:, 2:], 2, kc, vc)  # cache prefix of 2
    rows = [(0, 0), (1, 3), (0, 3)]
    yr, kn, vn = oracle.block_forward_rows(cfg, w, x[:, 2:], 2, kc, vc, rows)
    np.testing.assert_allclose(yr, np.stack([y[b, s] for b, s in rows]), atol=1e-12)
    np.testing.assert_allclose(kn, kfull[:, :, 2:6], atol=1e-13)
    np.testing.assert_allclose(vn, vfull[:, :, 2:6], atol=1e-13)


def test_stack_zero_blocks_is_norm_then_head():
    cfg = TINY
    vocab = 11
    emb = _rng("st_e", (vocab, 64))
    head = _rng("st_h", (vocab, 64))
    gfin = _rng("st_g", (64,), std=0.1, mean=1.0)
    toks = np.array([[3, 0, 10]])
    logits, _ = oracle.stack_forward(cfg, [], emb, gfin, head, toks, 0, [])
    for s, t in enumerate(toks[0]):
        e = emb[t]
        n = e / math.sqrt(float(np.mean(e ** 2)) + 1e-5) * gfin
        np.testing.assert_allclose(logits[0, s], head @ n, atol=1e-12)


# ------------------------------------------------- mixture of experts -------

MOE = dict(TINY, n_experts=6, top_k=2, d_ff=32, d_ff_shared=48)


def _moe_weights(cfg, tag):
    return {n: _rng(tag + n, s, std=0.1, mean=1.0) if n.endswith("norm") else _rng(tag + n, s, std=0.2)
            for n, s in synth.weight_shapes(**cfg).items()}


def test_moe_single_expert_without_shared_is_the_dense_ffn():
    cfg = dict(MOE, n_experts=1, top_k=1, d_ff_shared=0)
    w = _moe_weights(cfg, "m1")
    v = _rng("m1v", (7, 64))
    np.testing.assert_allclose(oracle.moe_ffn(cfg, w, v),
                               oracle.swiglu(v, w["w_gate"][0], w["w_up"][0], w["w_down"][0]), rtol=0, atol=1e-12)
    # and inside a whole block: equal to the dense block with that expert's weights
    dense = {k: (v_[0] if k in ("w_gate", "w_up", "w_down") else v_) for k, v_ in w.items() if k != "router"}
    wd, x, kc, vc = _tiny_inputs(TINY, B=1, S=5, Lmax=8, tag="m1b")
    wd.update(dense)
    wm = dict(wd, router=w["router"], w_gate=w["w_gate"], w_up=w["w_up"], w_down=w["w_down"])
    y_dense, _, _ = oracle.block_forward(dict(TINY, d_ff=32), wd, x, 0, kc, vc)
    y_moe, _, _ = oracle.block_forward(cfg, wm, x, 0, kc, vc)
    np.testing.assert_allclose(y_moe, y_dense, rtol=0, atol=1e-12)


def test_moe_identical_experts_make_routing_irrelevant():
    cfg = dict(MOE, d_ff_shared=0)
    w = _moe_weights(cfg, "mi")
    for n in ("w_gate", "w_up", "w_down"):
        w[n] = np.repeat(w[n][:1], cfg["n_experts"], axis=0)
    v = _rng("miv", (9, 64))
    np.testing.assert_allclose(oracle.moe_ffn(cfg, w, v),
                               oracle.swiglu(v, w["w_gate"][0], w["w_up"][0], w["w_down"][0]), rtol=0, atol=1e-12)


def test_moe_matches_bruteforce_top_k_with_shared_expert():
    cfg = MOE
    w = _moe_weights(cfg, "mb")
    v = _rng("mbv", (11, 64))
    out = oracle.moe_ffn(cfg, w, v)
    E, k = cfg["n_experts"], cfg["top_k"]
    for t in range(v.shape[0]):
        logits = [float(np.dot(w["router"][e], v[t])) for e in range(E)]
        chosen = []
        for _ in range(k):  # repeated arg-max, lowest id first among equals
            best = None
            for e in range(E):
                if e not in chosen and (best is None or logits[e] > logits[best]):
                    best = e
            chosen.append(best)
        ex = [math.exp(logits[e] - logits[chosen[0]]) for e in chosen]
        ref = np.zeros(64)
        for e, a in zip(chosen, ex):
            h = np.array([float(np.dot(w["w_gate"][e][f], v[t])) for f in range(cfg["d_ff"])])
            u = np.array([float(np.dot(w["w_up"][e][f], v[t])) for f in range(cfg["d_ff"])])
            ref += a / sum(ex) * (w["w_down"][e] @ (h / (1 + np.exp(-h)) * u))
        hs = w["shared_gate"] @ v[t]
        ref += w["shared_down"] @ (hs / (1 + np.exp(-hs)) * (w["shared_up"] @ v[t]))
        np.testing.assert_allclose(out[t], ref, rtol=0, atol=1e-11)


def test_moe_is_invariant_to_renumbering_the_experts():
    cfg = MOE
    w = _moe_weights(cfg, "mp")
    v = _rng("mpv", (13, 64))
    perm = np.array([3, 0, 5, 1, 4, 2])
    wp = dict(w)
    for n in ("w_gate", "w_up", "w_down", "router"):
        wp[n] = w[n][perm]
    np.testing.assert_allclose(oracle.moe_ffn(cfg, wp, v), oracle.moe_ffn(cfg, w, v), rtol=0, atol=1e-12)


def test_moe_with_every_expert_chosen_is_the_full_softmax_mixture():
    cfg = dict(MOE, top_k=6, d_ff_shared=0)
    w = _moe_weights(cfg, "ma")
    v = _rng("mav", (5, 64))
    logits = v @ w["router"].T
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ref = sum(p[:, e:e + 1] * oracle.swiglu(v, w["w_gate"][e], w["w_up"][e], w["w_down"][e]) for e in range(6))
    np.testing.assert_allclose(oracle.moe_ffn(cfg, w, v), ref, rtol=0, atol=1e-12)


def test_moe_router_ties_pick_the_lowest_id_and_weights_sum_to_one():
    cfg = dict(MOE, top_k=1)
    w = _moe_weights(cfg, "mt")
    w["router"][5] = w["router"][2]  # experts 2 and 5 always tie
    w["router"][[0, 1, 3, 4]] *= 0.0
    v = np.abs(_rng("mtv", (4, 64)))
    v = v * np.sign(w["router"][2])[None, :]  # positive logits for 2 and 5, zero for the rest
    ids, wts, _ = oracle.moe_route(cfg, w, v)
    assert ids.ravel().tolist() == [2, 2, 2, 2]
    np.testing.assert_allclose(wts, 1.0)
    ids2, wts2, _ = oracle.moe_route(MOE, dict(w), v)
    assert ids2.tolist() == [[2, 5]] * 4
    np.testing.assert_allclose(wts2.sum(-1), 1.0, rtol=1e-15)


def test_moe_shared_expert_alone_when_routed_outputs_vanish():
    cfg = MOE
    w = _moe_weights(cfg, "ms")
    w["w_down"] = np.zeros_like(w["w_down"])
    v = _rng("msv", (6, 64))
    np.testing.assert_allclose(oracle.moe_ffn(cfg, w, v),
                               oracle.swiglu(v, w["shared_gate"], w["shared_up"], w["shared_down"]),
                               rtol=0, atol=1e-12)


# ------------------------------------------------- greedy generation --------

def _identity_stack(cfg, n_layers, tag):
    """Blocks whose output projections vanish (y = x) around random attention
    and FFN weights, so the stack is embedding -> final norm -> head."""
    layers = []
    for l in range(n_layers):
        w = _tiny_weights(cfg, f"{tag}{l}")
        w["wo"] = np.zeros_like(w["wo"])
        w["w_down"] = np.zeros_like(w["w_down"])
        layers.append(w)
    return layers


def _one_hot_model(cfg, vocab, perm, scale=3.0):
    """One-hot embeddings e_t * scale and head rows head[j] = e_perm[j]: the
    logits of token t are sqrt(d)-scaled indicators of perm[j] == t, so the
    next token is the j with perm[j] == t."""
    d = cfg["d_model"]
    emb = np.zeros((vocab, d))
    emb[np.arange(vocab), np.arange(vocab)] = scale
    head = np.zeros((vocab, d))
    head[np.arange(vocab), np.asarray(perm)] = 1.0
    return emb, head


def test_greedy_generate_follows_the_closed_form_chain():
    cfg = TINY
    vocab, n_new, S, L = 13, 6, 4, 16
    perm = synth.uniform_int(0, "pins/perm", (vocab,), 1 << 30).argsort()  # a fixed permutation
    inv = np.argsort(perm)  # token t -> the j with perm[j] == t
    emb, head = _one_hot_model(cfg, vocab, perm)
    layers = _identity_stack(cfg, 2, "gg")
    prompt = np.array([[1, 5, 2, 7], [0, 0, 12, 3]])
    G, D = cfg["n_kv_heads"], cfg["d_model"] // cfg["n_heads"]
    caches = [(np.zeros((2, G, L, D)), np.zeros((2, G, L, D))) for _ in layers]
    toks, last, new = oracle.greedy_generate(cfg, layers, emb, np.ones(cfg["d_model"]), head, prompt, 3, caches, n_new)
    for b in range(2):
        t = prompt[b, -1]
        for i in range(n_new):
            t = inv[t]
            assert toks[b, i] == t
    # the last chosen token is not run: positions 3 .. 3 + S + n_new - 2 are cached, nothing after
    for kc, vc in new:
        assert np.all(np.abs(kc[:, :, 3:3 + S + n_new - 1]).sum(-1) > 0)
        assert np.all(kc[:, :, :3] == 0) and np.all(kc[:, :, 3 + S + n_new - 1:] == 0)
    # last logits: sqrt(d)-scaled indicator of the chosen token's preimage
    assert np.all(np.argmax(last, -1) == toks[:, -1])


def test_greedy_generate_breaks_ties_towards_the_lowest_id():
    cfg = TINY
    vocab = 9
    emb = _rng("tie_e", (vocab, cfg["d_model"]))
    layers = _identity_stack(cfg, 1, "tie")
    G, D = cfg["n_kv_heads"], cfg["d_model"] // cfg["n_heads"]
    caches = [(np.zeros((1, G, 8, D)), np.zeros((1, G, 8, D)))]
    toks, _, _ = oracle.greedy_generate(cfg, layers, emb, np.ones(64), np.zeros((vocab, 64)), np.array([[4, 2]]), 0,
                                        caches, 3)
    assert toks.tolist() == [[0, 0, 0]]
    head = np.zeros((vocab, 64))
    head[[3, 7]] = emb[5]  # rows 3 and 7 tie for token 5's successor
    toks, _, _ = oracle.greedy_generate(cfg, layers, emb, np.ones(64), head, np.array([[5]]), 0, caches, 1)
    assert toks.tolist() == [[3]]


def test_greedy_generate_equals_teacher_forced_argmax():
    # incremental decoding with the cache == one-shot forward over prompt + generated tokens
    cfg = TINY
    vocab, S, n_new, L = 23, 5, 4, 12
    layers = [_tiny_weights(cfg, f"tf{l}") for l in range(2)]
    emb = _rng("tf_e", (vocab, 64))
    head = _rng("tf_h", (vocab, 64))
    gfin = _rng("tf_g", (64,), std=0.1, mean=1.0)
    prompt = synth.uniform_int(0, "pins/tf_prompt", (2, S), vocab)
    G, D = cfg["n_kv_heads"], 16
    fresh = lambda: [(np.zeros((2, G, L, D)), np.zeros((2, G, L, D))) for _ in layers]
    toks, last, _ = oracle.greedy_generate(cfg, layers, emb, gfin, head, prompt, 1, fresh(), n_new)
    seq = np.concatenate([prompt, toks[:, :-1]], 1)
    logits, _ = oracle.stack_forward(cfg, layers, emb, gfin, head, seq, 1, fresh())
    np.testing.assert_array_equal(np.argmax(logits[:, S - 1:], -1), toks)
    np.testing.assert_allclose(last, logits[:, -1], rtol=0, atol=1e-10)
    assert len(set(toks.ravel().tolist())) > 1  # not a degenerate chain


# ------------------------------------------------- printed counts ------------

def test_kv_cache_counts_match_printed_values():
    g = GOLDEN["kv_cache_counts"]
    assert oracle.kv_values_per_token(1, 8, 128) == g["llama3_8b_per_layer_values"]
    assert oracle.kv_values_per_token(1, 32, 128) == g["llama3_8b_per_layer_values_mha"]
    assert oracle.kv_values_per_token(32, 8, 128) == g["llama3_8b_32_layers_values"]
    assert oracle.kv_values_per_token(32, 8, 128) * 2 // 1024 == g["llama3_8b_bytes_per_token_16bit_KB"]
    assert abs(oracle.kv_values_per_token(32, 8, 128) * 2 * 8192 / 2 ** 30 - g["llama3_8b_8192_tokens_GB_approx"]) < 0.01
    assert oracle.kv_values_per_token(30, 3, 64) == g["smollm2_values_per_token"]
    assert oracle.kv_values_per_token(30, 9, 64) == g["smollm2_values_per_token_mha"]
    assert oracle.kv_values_per_token(12, 12, 64) == g["gpt2_small_values_per_token"]
    b = oracle.kv_values_per_token(32, 8, 128) * 2
    assert round(b / 1000) == g["llama31_8b_bytes_per_token_KB"]
    assert round(b * 131072 / 1e9, 1) == g["llama31_8b_cache_GB_at_131072"]
    assert round(4 * b * 131072 / 1e9, 1) == g["llama31_8b_cache_GB_at_131072_mha"]


def test_param_counts_match_printed_values():
    g = GOLDEN["param_counts"]
    blk = oracle.block_param_count(4096, 32, 8, 14336)
    assert round(blk["total"] / 1e6) == g["llama3_8b_block_millions"]
    assert round(blk["ffn"] / 1e6) == g["llama3_8b_ffn_millions"]
    assert round(100 * blk["ffn"] / blk["total"]) == g["llama3_8b_ffn_share_percent"]
    mha = oracle.block_param_count(4096, 32, 32, 14336)
    assert round(100 * mha["ffn"] / mha["total"]) == g["llama3_8b_ffn_share_mha_percent"]
    sm = oracle.block_param_count(576, 9, 3, 1536)
    assert round(100 * sm["ffn"] / sm["total"]) == g["smollm2_ffn_share_percent"]
    assert round(oracle.model_param_count(576, 9, 3, 1536, 30, 49152, tied=True) / 1e6, 1) == g["smollm2_params_millions"]
    assert round(oracle.model_param_count(576, 9, 9, 1536, 30, 49152, tied=True) / 1e6, 1) == g["smollm2_params_mha_millions"]
    n8b = oracle.model_param_count(4096, 32, 8, 14336, 32, 128256, tied=False)
    assert round(n8b / 1e9, 1) == g["llama3_8b_params_billions"]
    assert round(n8b * 2 / 1e9, 1) == g["llama31_8b_weights_GB_bf16"]


# --------------------------------------------------- plants (negative) -------

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant typical slips in the oracle (on the CPU) and check a pin fails."""
    import oracle.llama_block as ob

    cfg = TINY
    # 1. wrong grouping index (tiling h % G instead of h // r)
    orig = ob.gqa_attention

    def tiled(q, kc, vc, sp):
        H = q.shape[2]
        G = kc.shape[1]
        perm = [h % G for h in range(H)]
        kc2 = np.stack([kc[:, g] for g in perm], 1)
        vc2 = np.stack([vc[:, g] for g in perm], 1)
        return orig(q, kc2, vc2, sp)

    w, x, kc, vc = _tiny_inputs(cfg, B=1, S=1, Lmax=2, tag="pl")
    y_ok, _, _ = ob.block_forward(cfg, w, x, 0, kc, vc)
    monkeypatch.setattr(ob, "gqa_attention", tiled)
    y_bad, _, _ = ob.block_forward(cfg, w, x, 0, kc, vc)
    monkeypatch.setattr(ob, "gqa_attention", orig)
    assert np.max(np.abs(y_bad - y_ok)) > 1e-3  # the single-token closed form catches it

    # 2. exponent i/D instead of 2i/D breaks the printed RoPE period
    f_bad = 1e5 ** (-np.arange(32) / 64)
    assert abs(2 * math.pi / f_bad.min() - 438000) > 1000

    # 3. eps outside the root breaks the eps-in-root closed form
    bad = np.ones(2) / (np.sqrt(1.0) + 3.0)
    assert not np.allclose(bad, oracle.rms_norm(np.ones(2), np.ones(2), 3.0))
