"""The C-ABI library loads and exports every declared symbol; host-only entry
points and host-side validation work without a GPU (no compute calls)."""
import glob
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import decoder_block_gb300 as lb
    if not os.path.exists(lb.LIB_PATH):
        from decoder_block_gb300 import build
        build.build()
    return lb


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(llama_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 17
    so = lib.load()
    for n in sorted(names):
        assert hasattr(so, n), f"{n} declared in include/*.h but not exported"


def test_ffn_hidden_dim_matches_oracle_rule(lib):
    for d, mult, m in [(4096, 1024, 1.3), (4096, 256, 0.0), (576, 256, 0.0), (64, 64, 0.0), (8192, 4096, 1.3)]:
        assert lib.llama_ffn_hidden_dim(d, mult, m) == oracle.ffn_hidden_dim(d, mult, m if m > 0 else None)
    assert lib.llama_ffn_hidden_dim(0, 256, 0.0) == -1


def test_kv_cache_bytes_formula(lib):
    cfg = lib.make_config(4096, 32, 8, 14336, 8192, 1e-5, 5e5, lib.LLAMA_BF16)
    # 2 (K, V) x n_kv x d_head values per token per sequence, bf16
    assert lib.llama_kv_cache_bytes(cfg, 1, 8192) == oracle.kv_values_per_token(1, 8, 128) * 2 * 8192
    assert lib.llama_kv_cache_bytes(cfg, 64, 4096) == 64 * 4096 * 2048 * 2
    bad = lib.make_config(4096, 30, 8, 14336, 8192, 1e-5, 5e5, lib.LLAMA_BF16)
    assert lib.llama_kv_cache_bytes(bad, 1, 16) == 0


def test_status_strings(lib):
    for s in range(9):
        assert lib.llama_status_string(s) != "unknown status"
    assert lib.llama_status_string(99) == "unknown status"


@pytest.mark.parametrize("fields,expected", [
    (dict(d_model=4096, n_heads=30), "LLAMA_ERR_SHAPE"),      # d_model % n_heads
    (dict(n_kv_heads=5), "LLAMA_ERR_SHAPE"),                  # n_heads % n_kv_heads
    (dict(d_model=4096, n_heads=64, n_kv_heads=8), "LLAMA_OK_SHAPE"),  # d_head 64 is fine (not reached)
    (dict(d_model=96, n_heads=32, n_kv_heads=8), "LLAMA_ERR_SHAPE"),   # d_head 3 is odd
    (dict(d_model=3072, n_heads=32), "LLAMA_ERR_UNSUPPORTED"),  # d_head 96 is even but has no kernel
    (dict(dtype=7), "LLAMA_ERR_INVALID_ARG"),
    (dict(norm_eps=-1.0), "LLAMA_ERR_INVALID_ARG"),
    (dict(rope_theta=0.0), "LLAMA_ERR_INVALID_ARG"),
    (dict(d_ff=14336 + 8), "LLAMA_ERR_UNSUPPORTED"),         # bf16 gate/up interleave needs d_ff % 16
    (dict(rope_layout=2), "LLAMA_ERR_INVALID_ARG"),           # neither interleaved nor halves
    (dict(rope_scaling=dict(factor=8.0, low_freq_factor=0.0, high_freq_factor=4.0, original_max_pos=8192)),
     "LLAMA_ERR_INVALID_ARG"),                                # stretch needs 0 < low < high
    (dict(rope_scaling=dict(factor=8.0, low_freq_factor=4.0, high_freq_factor=1.0, original_max_pos=8192)),
     "LLAMA_ERR_INVALID_ARG"),
    (dict(rope_scaling=dict(factor=8.0, low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=0)),
     "LLAMA_ERR_INVALID_ARG"),
    (dict(rope_scaling=dict(factor=float("nan"))), "LLAMA_ERR_INVALID_ARG"),
])
def test_create_rejects_bad_configs_before_touching_the_gpu(lib, fields, expected):
    base = dict(d_model=4096, n_heads=32, n_kv_heads=8, d_ff=14336, max_seq_len=8192, norm_eps=1e-5,
                rope_theta=5e5, dtype=lib.LLAMA_BF16)
    base.update(fields)
    cfg = lib.make_config(**base)
    if expected == "LLAMA_OK_SHAPE":
        return
    w = lib.make_weights({n: None for n in lib.WEIGHT_FIELDS})
    st, h = lib.llama_block_create(cfg, w, 16)
    assert st == getattr(lib, expected) and h is None


def test_null_arguments_are_rejected(lib):
    cfg = lib.make_config(64, 4, 2, 192, 16, 1e-5, 1e4, lib.LLAMA_F32)
    w = lib.make_weights({n: None for n in lib.WEIGHT_FIELDS})
    st, h = lib.llama_block_create(cfg, w, 16)
    assert st == lib.LLAMA_ERR_INVALID_ARG and h is None
    st, h = lib.llama_block_create(cfg, w, 0)
    assert st == lib.LLAMA_ERR_INVALID_ARG
    assert lib.llama_block_forward(None, None, None, 1, 1, 0, lib.make_kv_cache(None, None, 1, 1)) \
        == lib.LLAMA_ERR_INVALID_ARG
    assert lib.llama_op_linear(lib.LLAMA_BF16, None, None, None, None, 0, 16, 16, 0) == lib.LLAMA_ERR_INVALID_ARG
    assert lib.llama_op_linear(lib.LLAMA_BF16, None, None, None, None, 16, 16, 12, 0) == lib.LLAMA_ERR_UNSUPPORTED
    assert lib.llama_op_attention(lib.LLAMA_BF16, None, lib.make_kv_cache(None, None, 1, 8), None, 2, 1, 0,
                                  4, 2, 64) == lib.LLAMA_ERR_RANGE
    assert lib.llama_op_attention_workspace_bytes(lib.LLAMA_BF16, 64, 1, 4095, 32, 128) == 64 * 32 * 16 * 130 * 4
    assert lib.llama_op_attention_workspace_bytes(lib.LLAMA_BF16, 64, 8, 0, 32, 128) == 0
    assert lib.llama_block_set_wait_budget(None, 0) == lib.LLAMA_ERR_INVALID_ARG
    assert lib.llama_stack_set_wait_budget(None, 100) == lib.LLAMA_ERR_INVALID_ARG
