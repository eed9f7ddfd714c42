"""Per-step parity of the CUDA kernels against the fp64 oracle (GPU)."""
import numpy as np
import pytest

import oracle
import synth
from _helpers import assert_parity, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lb():
    import decoder_block_gb300 as m
    m.load()
    return m


def _bf16(tag, shape, std=1.0):
    return synth.f32_to_bf16_bits(synth.normal(0, "ops/" + tag, shape, std=std))


# ------------------------------------------------------------------ GEMM ---

GEMM_SHAPES = [
    (128, 256, 64),      # exactly one tile, one K step
    (1, 16, 8),          # degenerate: one row, K shorter than a K step
    (127, 200, 72),      # ragged M, N and K tails
    (300, 960, 576),     # SmolLM2 QKV width, K = 9 K steps
    (257, 264, 136),
    (64, 6144, 4096),    # decode-sized M, Llama-3-8B QKV
    (1000, 1536, 512),
    (2000, 4000, 4104),  # CTA-pair tiles (residual and fp32 epilogues): ragged M, N and K
    (1024, 4864, 1032),  # exactly one wave of pair tiles (76 pairs), K tail
    (1000, 4864, 1032),  # the same with a ragged last pair tile (232 live rows)
    (768, 5000, 512),    # just under one wave of pair tiles: single-CTA tiles
    (4096, 1280, 2048),  # a plan with a split tail on single CTAs, whole tiles on pairs
    (3000, 2000, 4104),  # ragged M, N, K on pairs, 12 x 8 pair tiles
]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_linear_bf16_tensor_core(lb, M, N, K, epi):
    A = _bf16(f"A{M}{N}{K}", (M, K))
    W = _bf16(f"W{M}{N}{K}", (N, K), std=0.05)
    R = _bf16(f"R{M}{N}{K}", (M, N))
    ref = oracle.linear(synth.as_f64(A), synth.as_f64(W))
    if epi == 1:
        ref = ref + synth.as_f64(R)
    a, w, r = to_dev(A), to_dev(W), to_dev(R)
    t = torch()
    c = t.empty((M, N), dtype=t.float32 if epi == 2 else t.bfloat16, device="cuda")
    lb.check(lb.llama_op_linear(lb.LLAMA_BF16, a, w, r if epi == 1 else None, c, M, N, K, epi))
    t.cuda.synchronize()
    got = to_f64(c)
    assert_parity(got, ref, "bf16", f"linear M={M} N={N} K={K} epi={epi}")
    if epi == 2:  # fp32 output: only accumulation-order error remains
        bound = 1e-5 * np.abs(synth.as_f64(A)) @ np.abs(synth.as_f64(W)).T + 1e-6
        assert np.all(np.abs(got - ref) <= bound)


def test_linear_residual_in_place(lb):
    M, N, K = 200, 512, 256
    A, W, R = _bf16("ipA", (M, K)), _bf16("ipW", (N, K), 0.05), _bf16("ipR", (M, N))
    ref = oracle.linear(synth.as_f64(A), synth.as_f64(W)) + synth.as_f64(R)
    a, w, r = to_dev(A), to_dev(W), to_dev(R)
    lb.check(lb.llama_op_linear(lb.LLAMA_BF16, a, w, r, r, M, N, K, 1))
    torch().cuda.synchronize()
    assert_parity(to_f64(r), ref, "bf16", "linear residual in place")


def test_linear_f32(lb):
    M, N, K = 37, 72, 40
    A = synth.normal(0, "ops/fA", (M, K))
    W = synth.normal(0, "ops/fW", (N, K), std=0.1)
    t = torch()
    c = t.empty((M, N), dtype=t.float32, device="cuda")
    lb.check(lb.llama_op_linear(lb.LLAMA_F32, to_dev(A), to_dev(W), None, c, M, N, K, 0))
    t.cuda.synchronize()
    assert_parity(to_f64(c), oracle.linear(A, W), "f32", "linear f32")


# --------------------------------------------------------------- RMSNorm ---

@pytest.mark.parametrize("T,d,dtype", [(1, 64, "f32"), (33, 576, "bf16"), (100, 4096, "bf16"), (7, 192, "f32")])
def test_rmsnorm(lb, T, d, dtype):
    x32 = synth.normal(0, f"ops/rx{T}{d}", (T, d), std=2.0)
    g32 = synth.normal(0, f"ops/rg{T}{d}", (d,), std=0.1, mean=1.0)
    conv = (lambda a: a) if dtype == "f32" else synth.f32_to_bf16_bits
    x, g = conv(x32), conv(g32)
    ref = oracle.rms_norm(synth.as_f64(x), synth.as_f64(g), 1e-5)
    xd, gd = to_dev(x), to_dev(g)
    out = torch().empty_like(xd)
    lb.check(lb.llama_op_rmsnorm(lb.LLAMA_BF16 if dtype == "bf16" else lb.LLAMA_F32, xd, gd, out, T, d, 1e-5))
    torch().cuda.synchronize()
    assert_parity(to_f64(out), ref, dtype, "rmsnorm")


# ------------------------------------------------------- RoPE + KV write ---

LLAMA31_SCALING = dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)


@pytest.mark.parametrize("B,S,start_pos,H,G,D,dtype,theta,layout,scaling", [
    (1, 16, 0, 4, 2, 16, "f32", 1e4, "interleaved", None),
    (3, 37, 5, 9, 3, 64, "bf16", 1e5, "interleaved", None),
    (2, 70, 4000, 32, 8, 128, "bf16", 5e5, "interleaved", None),
    (1, 16, 3, 4, 2, 16, "f32", 1e4, "halves", None),
    (3, 37, 5, 9, 3, 64, "bf16", 1e5, "halves", None),
    (2, 9, 20000, 8, 2, 128, "bf16", 5e5, "halves", LLAMA31_SCALING),
    (1, 12, 30000, 4, 2, 128, "f32", 5e5, "interleaved", LLAMA31_SCALING),
])
def test_rope_kv_write(lb, B, S, start_pos, H, G, D, dtype, theta, layout, scaling):
    t = torch()
    conv = (lambda a: a) if dtype == "f32" else synth.f32_to_bf16_bits
    L = start_pos + S + 3
    qkv = conv(synth.normal(0, "ops/qkv", (B * S, (H + 2 * G) * D)))
    k0 = conv(synth.normal(0, "ops/k0", (B + 1, G, L, D)))
    v0 = conv(synth.normal(0, "ops/v0", (B + 1, G, L, D)))
    table = t.empty((L, D // 2, 2), dtype=t.float32, device="cuda")
    lb.check(lb.llama_op_rope_table(table, L, D, theta, scaling))
    qd, kd, vd = to_dev(qkv), to_dev(k0), to_dev(v0)
    q_out = t.empty((B * S, H * D), dtype=qd.dtype, device="cuda")
    kv = lb.make_kv_cache(kd, vd, B + 1, L)
    dt = lb.LLAMA_BF16 if dtype == "bf16" else lb.LLAMA_F32
    lcode = lb.LLAMA_ROPE_HALVES if layout == "halves" else lb.LLAMA_ROPE_INTERLEAVED
    lb.check(lb.llama_op_rope_kv_write(dt, qd, q_out, kv, table, L, B, S, start_pos, H, G, D, lcode))
    t.cuda.synchronize()
    x = synth.as_f64(qkv).reshape(B, S, H + 2 * G, D)
    pos = start_pos + np.arange(S)
    q_ref = oracle.rope(x[:, :, :H], pos, theta, layout, scaling)
    k_ref = oracle.rope(x[:, :, H:H + G], pos, theta, layout, scaling)
    v_ref = x[:, :, H + G:]
    assert_parity(to_f64(q_out).reshape(B, S, H, D), q_ref, dtype, "rotated q")
    kg, vg = to_f64(kd), to_f64(vd)
    assert_parity(kg[:B, :, start_pos:start_pos + S].transpose(0, 2, 1, 3), k_ref, dtype, "K cache slice")
    np.testing.assert_array_equal(vg[:B, :, start_pos:start_pos + S].transpose(0, 2, 1, 3), v_ref)
    # everything outside the written slice is bit-for-bit unchanged
    kb, vb = synth.as_f64(k0), synth.as_f64(v0)
    mask = np.ones(kb.shape, dtype=bool)
    mask[:B, :, start_pos:start_pos + S] = False
    np.testing.assert_array_equal(kg[mask], kb[mask])
    np.testing.assert_array_equal(vg[mask], vb[mask])
    # the table itself: fp32 rounding of cos/sin of the exact angle
    tab = table.cpu().numpy().astype(np.float64)
    ang = np.arange(L)[:, None] * oracle.rope_frequencies(D, theta, scaling)[None, :]
    assert np.max(np.abs(tab[..., 0] - np.cos(ang))) < 1e-6
    assert np.max(np.abs(tab[..., 1] - np.sin(ang))) < 1e-6


# ------------------------------------------------------------- attention ---

ATTN_CASES = [
    # B, S, start_pos, H, G, D, dtype
    (1, 16, 0, 4, 2, 16, "f32"),
    (2, 33, 0, 4, 4, 64, "bf16"),     # MHA (n_rep 1), ragged S
    (3, 45, 7, 9, 3, 64, "bf16"),     # SmolLM2 grouping (n_rep 3), cache prefix
    (1, 200, 0, 8, 2, 128, "bf16"),   # n_rep 4, several key tiles
    (2, 130, 60, 4, 2, 128, "bf16"),  # prefix + ragged
    (2, 70, 5, 10, 2, 128, "bf16"),   # n_rep 5: 24 positions x 5 heads per 128-row query tile
    (1, 300, 0, 40, 8, 128, "bf16"),  # Llama-4-Scout grouping (n_rep 5), several key tiles
    (1, 50, 0, 12, 2, 64, "bf16"),    # n_rep 6: 16 positions per tile, 32 rows left zero
    (1, 90, 11, 14, 2, 128, "bf16"),  # n_rep 7: 16 positions, 112 live rows, cache prefix
    (2, 100, 3, 6, 2, 64, "bf16"),    # n_rep 3: 40 positions per tile (120 rows)
    # D = 128 prefill edge cases: a single key tile, a one-key last tile, MHA, n_rep 8, a long cached prefix
    (1, 64, 0, 8, 2, 128, "bf16"),    # one key tile, half of it past the end; one query block
    (1, 129, 0, 32, 8, 128, "bf16"),  # Llama-3-8B grouping; the last key tile holds one key
    (2, 257, 100, 16, 16, 128, "bf16"),  # MHA (128 positions per query tile), cache prefix
    (1, 100, 0, 16, 2, 128, "bf16"),  # n_rep 8: 16 positions per tile
    (1, 600, 1500, 32, 8, 128, "bf16"),  # a chunk after a long cached prefix (17 key tiles)
    (3, 2, 5, 8, 2, 128, "bf16"),     # two-position prefill
    (5, 1, 300, 8, 2, 128, "bf16"),   # decode step, S = 1, two key chunks
    (3, 1, 77, 9, 3, 64, "bf16"),     # decode, one chunk, n_rep 3
    (2, 1, 1000, 32, 8, 128, "bf16"), # decode, ragged last chunk
    (4, 1, 0, 4, 4, 64, "bf16"),      # decode of the first position (MHA)
    (1, 1, 700, 16, 2, 128, "bf16"),  # decode, n_rep 8
    (3, 1, 5, 8, 2, 128, "bf16"),     # decode over 6 cached positions (one partial tile)
    (1, 1, 40, 8, 2, 128, "bf16"),    # decode with fewer query rows than one 16-row operand
    (2, 1, 600, 4, 4, 128, "bf16"),   # decode, MHA, d_head 128
    (2, 1, 2047, 32, 8, 128, "bf16"), # decode, chunk edge (2048 cached positions)
    (2, 1, 900, 32, 2, 128, "bf16"),  # decode, n_rep 16 (all sixteen head columns live)
    (3, 1, 520, 24, 4, 128, "bf16"),  # decode, n_rep 6 (eight-column softmax, two padded)
    (2, 3, 0, 2, 1, 32, "bf16"),
]


@pytest.mark.parametrize("B,S,start_pos,H,G,D,dtype", ATTN_CASES)
def test_attention(lb, B, S, start_pos, H, G, D, dtype):
    t = torch()
    conv = (lambda a: a) if dtype == "f32" else synth.f32_to_bf16_bits
    L = start_pos + S + 5
    q = conv(synth.normal(0, "ops/aq", (B, S, H, D)))
    kc = conv(synth.normal(0, "ops/ak", (B, G, L, D)))
    vc = conv(synth.normal(0, "ops/av", (B, G, L, D)))
    ref = oracle.gqa_attention(synth.as_f64(q), synth.as_f64(kc), synth.as_f64(vc), start_pos)
    qd, kd, vd = to_dev(q), to_dev(kc), to_dev(vc)
    o = t.empty_like(qd)
    dt = lb.LLAMA_BF16 if dtype == "bf16" else lb.LLAMA_F32
    nws = lb.llama_op_attention_workspace_bytes(dt, B, S, start_pos, H, D)
    ws = t.empty(max(nws, 16), dtype=t.uint8, device="cuda")
    lb.check(lb.llama_op_attention(dt, qd, lb.make_kv_cache(kd, vd, B, L), o, B, S, start_pos, H, G, D, ws, nws))
    t.cuda.synchronize()
    assert_parity(to_f64(o), ref, dtype, f"attention B={B} S={S} sp={start_pos} H={H} G={G} D={D}")


# Keys whose scale grows with their position, (1 + p/8): each 32-key chunk's
# largest score tends to exceed the running maximum by more than 2^8 (in
# log2 units), so the online softmax raises its maximum inside a key tile and
# rescales the probabilities already written for that tile, the row sum and O.
GROWING_CASES = [
    # B, S, start_pos, H, G, D
    (1, 200, 0, 8, 2, 128),
    (2, 130, 60, 4, 2, 128),
    (1, 90, 11, 14, 2, 128),
    (3, 45, 7, 9, 3, 64),
]


@pytest.mark.parametrize("B,S,start_pos,H,G,D", GROWING_CASES)
def test_attention_growing_scores(lb, B, S, start_pos, H, G, D):
    t = torch()
    L = start_pos + S + 5
    ramp = (1.0 + np.arange(L, dtype=np.float32) / 8.0)[None, None, :, None]
    q = synth.f32_to_bf16_bits(synth.normal(0, "ops/gq", (B, S, H, D)))
    kc = synth.f32_to_bf16_bits(synth.normal(0, "ops/gk", (B, G, L, D)) * ramp)
    vc = synth.f32_to_bf16_bits(synth.normal(0, "ops/gv", (B, G, L, D)))
    ref = oracle.gqa_attention(synth.as_f64(q), synth.as_f64(kc), synth.as_f64(vc), start_pos)
    qd, kd, vd = to_dev(q), to_dev(kc), to_dev(vc)
    o = t.empty_like(qd)
    nws = lb.llama_op_attention_workspace_bytes(lb.LLAMA_BF16, B, S, start_pos, H, D)
    ws = t.empty(max(nws, 16), dtype=t.uint8, device="cuda")
    lb.check(lb.llama_op_attention(lb.LLAMA_BF16, qd, lb.make_kv_cache(kd, vd, B, L), o, B, S, start_pos, H, G, D,
                                   ws, nws))
    t.cuda.synchronize()
    assert_parity(to_f64(o), ref, "bf16", f"attention, growing keys, B={B} S={S} sp={start_pos} H={H} G={G} D={D}")
