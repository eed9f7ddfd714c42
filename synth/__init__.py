"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only *draws numbers*: it holds none of the decoder block's
arithmetic.  Both sides of every parity check (the CUDA library and the fp64
oracle) consume the arrays produced here, so a difference between them can
only come from the arithmetic each side does.

Generator (counter based, so any slice can be drawn on its own):
  * key      = SplitMix64(seed * 0x9E3779B97F4A7C15 + FNV-1a-64(tag))
  * word[n]  = SplitMix64 finaliser of (key + (n + 1) * 0x9E3779B97F4A7C15)
  * normals  : Box-Muller on the two 32-bit halves of word[n // 2]
               (u1 = (hi + 1) / 2^32 in (0, 1], u2 = lo / 2^32), element 2m takes
               the cosine branch and 2m + 1 the sine branch; radius in fp64, the
               angle's cosine/sine in fp32, product rounded once to fp32.
  * bf16     : round-to-nearest-even of those fp32 values (bit manipulation).
  * integers : multiply-shift of the 64-bit word onto [0, high).

SplitMix64 is Steele, Lea and Flood, "Fast splittable pseudorandom number
generators" (OOPSLA 2014); Box-Muller is Box and Muller (1958).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _fnv1a64(tag: str) -> int:
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _mix_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int."""
    m = 0xFFFFFFFFFFFFFFFF
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_key(seed: int, tag: str) -> int:
    return _mix_int(seed * 0x9E3779B97F4A7C15 + _fnv1a64(tag) + 0x9E3779B97F4A7C15)


def _words(key: int, start: int, count: int, out: np.ndarray | None = None,
           tmp: np.ndarray | None = None) -> np.ndarray:
    """word[start .. start + count) of the stream with the given key (uint64)."""
    z = np.empty(count, dtype=np.uint64) if out is None else out[:count]
    t = np.empty(count, dtype=np.uint64) if tmp is None else tmp[:count]
    with np.errstate(over="ignore"):
        z[:] = _counter_base(count)
        z += np.uint64(start + 1)
        z *= _GOLDEN
        z += np.uint64(key)
        # SplitMix64 finaliser, in place
        np.right_shift(z, np.uint64(30), out=t)
        z ^= t
        z *= _M1
        np.right_shift(z, np.uint64(27), out=t)
        z ^= t
        z *= _M2
        np.right_shift(z, np.uint64(31), out=t)
        z ^= t
    return z


_BASE = np.zeros(0, dtype=np.uint64)


def _counter_base(count: int) -> np.ndarray:
    global _BASE
    if _BASE.size < count:
        _BASE = np.arange(max(count, _CHUNK), dtype=np.uint64)
    return _BASE[:count]


def _normal_chunks(key: int, out: np.ndarray, total: int, p_begin: int, p_end: int, std: float, mean: float):
    """Fill out[2*p_begin : 2*p_end] (clipped to total) with the normals of pairs [p_begin, p_end)."""
    n = min(_CHUNK, max(p_end - p_begin, 1))
    wbuf = np.empty(n, dtype=np.uint64)
    tbuf = np.empty(n, dtype=np.uint64)
    rad = np.empty(n, dtype=np.float64)
    ang = np.empty(n, dtype=np.float32)
    trig = np.empty(n, dtype=np.float32)
    z = np.empty((n, 2), dtype=np.float64)
    for p0 in range(p_begin, p_end, _CHUNK):
        c = min(p_end, p0 + _CHUNK) - p0
        w = _words(key, p0, c, wbuf, tbuf)
        r = rad[:c]
        np.right_shift(w, np.uint64(32), out=tbuf[:c])
        r[:] = tbuf[:c]
        r += 1.0
        r *= 1.0 / 4294967296.0  # u1 in (0, 1]
        np.log(r, out=r)
        r *= -2.0
        np.sqrt(r, out=r)  # Box-Muller radius
        w &= np.uint64(0xFFFFFFFF)
        a = ang[:c]
        a[:] = w
        a *= np.float32(2.0 * np.pi / 4294967296.0)  # angle 2 pi u2
        zc = z[:c]
        np.cos(a, out=trig[:c])
        zc[:, 0] = trig[:c]
        np.sin(a, out=trig[:c])
        zc[:, 1] = trig[:c]
        zc *= r[:, None]
        if std != 1.0:
            zc *= std
        if mean != 0.0:
            zc += mean
        e0 = 2 * p0
        e1 = min(total, 2 * (p0 + c))
        out[e0:e1] = zc.reshape(-1)[: e1 - e0]


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures
        import os
        _POOL = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def normal(seed: int, tag: str, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """fp32 array of N(mean, std^2) samples for the stream (seed, tag).

    Large arrays are filled by several host threads; every element depends
    only on (seed, tag, index), so the result does not depend on the split."""
    shape = tuple(int(s) for s in np.atleast_1d(shape)) if not isinstance(shape, tuple) else shape
    total = int(np.prod(shape, dtype=np.int64))
    key = stream_key(seed, tag)
    out = np.empty(total, dtype=np.float32)
    npairs = (total + 1) // 2
    if npairs <= 4 * _CHUNK:
        _normal_chunks(key, out, total, 0, npairs, std, mean)
    else:
        step = 4 * _CHUNK
        futs = [_pool().submit(_normal_chunks, key, out, total, p, min(npairs, p + step), std, mean)
                for p in range(0, npairs, step)]
        for f in futs:
            f.result()
    return out.reshape(shape)


def uniform_int(seed: int, tag: str, shape, high: int) -> np.ndarray:
    """int32 array uniform on [0, high) (multiply-shift of the high 32 bits)."""
    shape = tuple(shape)
    total = int(np.prod(shape, dtype=np.int64))
    w = _words(stream_key(seed, tag), 0, total)
    hi = w >> np.uint64(32)
    v = (hi * np.uint64(high)) >> np.uint64(32)
    return v.astype(np.int32).reshape(shape)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# Workload shapes (Llama block configurations) and their input recipes.
# ---------------------------------------------------------------------------

SHAPES = {
    # name: model dims, batch/sequence and start position
    "tiny_f32": dict(d_model=64, n_heads=4, n_kv_heads=2, d_ff=192, norm_eps=1e-5, rope_theta=1e4,
                     dtype="f32", B=1, S=16, start_pos=0, max_seq_len=16),
    "smollm2_135m": dict(d_model=576, n_heads=9, n_kv_heads=3, d_ff=1536, norm_eps=1e-5, rope_theta=1e5,
                         dtype="bf16", B=8, S=1024, start_pos=0, max_seq_len=1024),
    "llama3_8b_prefill_b1s8192": dict(d_model=4096, n_heads=32, n_kv_heads=8, d_ff=14336, norm_eps=1e-5,
                                      rope_theta=5e5, dtype="bf16", B=1, S=8192, start_pos=0, max_seq_len=8192),
    "llama3_8b_prefill_b4s2048": dict(d_model=4096, n_heads=32, n_kv_heads=8, d_ff=14336, norm_eps=1e-5,
                                      rope_theta=5e5, dtype="bf16", B=4, S=2048, start_pos=0, max_seq_len=2048),
    "llama3_8b_decode_b64": dict(d_model=4096, n_heads=32, n_kv_heads=8, d_ff=14336, norm_eps=1e-5,
                                 rope_theta=5e5, dtype="bf16", B=64, S=1, start_pos=4095, max_seq_len=4096),
}

WEIGHT_NAMES = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def weight_shapes(d_model, n_heads, n_kv_heads, d_ff, n_experts=0, d_ff_shared=0, **_):
    """Parameter shapes of one block.  With n_experts > 0 the feed-forward is a
    mixture of experts: w_gate / w_up / w_down stacked per expert, a router
    [n_experts, d_model] and, when d_ff_shared > 0, a shared expert."""
    dh = d_model // n_heads
    out = {
        "attn_norm": (d_model,),
        "wq": (n_heads * dh, d_model),
        "wk": (n_kv_heads * dh, d_model),
        "wv": (n_kv_heads * dh, d_model),
        "wo": (d_model, n_heads * dh),
        "ffn_norm": (d_model,),
        "w_gate": (d_ff, d_model),
        "w_up": (d_ff, d_model),
        "w_down": (d_model, d_ff),
    }
    if n_experts:
        out["w_gate"] = (n_experts, d_ff, d_model)
        out["w_up"] = (n_experts, d_ff, d_model)
        out["w_down"] = (n_experts, d_model, d_ff)
        out["router"] = (n_experts, d_model)
        if d_ff_shared:
            out["shared_gate"] = (d_ff_shared, d_model)
            out["shared_up"] = (d_ff_shared, d_model)
            out["shared_down"] = (d_model, d_ff_shared)
    return out


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 samples in the storage type: fp32 as is, bf16 as uint16 bit patterns."""
    return a32 if dtype == "f32" else f32_to_bf16_bits(a32)


def as_f64(a: np.ndarray) -> np.ndarray:
    """Exact fp64 value of a stored array (fp32, or bf16 bit patterns)."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def block_weights(shape: dict, seed: int = 0, layer: int = 0) -> dict:
    """Linear weights ~ N(0, 0.02^2), RMSNorm gains ~ 1 + N(0, 0.1^2), no biases."""
    dt = shape["dtype"]
    out = {}
    for name, shp in weight_shapes(**shape).items():
        tag = f"L{layer}/{name}"
        if name.endswith("norm"):
            out[name] = _store(normal(seed, tag, shp, std=0.1, mean=1.0), dt)
        else:
            out[name] = _store(normal(seed, tag, shp, std=0.02), dt)
    return out


def block_activations(shape: dict, seed: int = 0, tag: str = "x", B=None, S=None) -> np.ndarray:
    """Block input x ~ N(0, 1), [B, S, d_model]."""
    B = shape["B"] if B is None else B
    S = shape["S"] if S is None else S
    return _store(normal(seed, tag, (B, S, shape["d_model"])), shape["dtype"])


def kv_cache(shape: dict, seed: int = 0, max_batch=None, max_seq_len=None, fill_upto: int = 0,
             layer: int = 0):
    """K and V caches [max_batch, n_kv, max_seq, d_head]; positions < fill_upto ~ N(0, 1), the rest 0."""
    mb = shape["B"] if max_batch is None else max_batch
    ms = shape["max_seq_len"] if max_seq_len is None else max_seq_len
    G = shape["n_kv_heads"]
    D = shape["d_model"] // shape["n_heads"]
    caches = []
    for which in ("k", "v"):
        c = np.zeros((mb, G, ms, D), dtype=np.float32)
        if fill_upto > 0:
            c[:, :, :fill_upto, :] = normal(seed, f"L{layer}/cache_{which}", (mb, G, fill_upto, D))
        caches.append(_store(c, shape["dtype"]))
    return caches[0], caches[1]
