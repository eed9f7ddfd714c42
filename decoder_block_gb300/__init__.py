"""Python binding of libllama_block.so (the GB300 Llama decoder-block library).

Argument marshalling only: every function here forwards to the C entry point of
the same name (include/llama_block.h, include/llama_ops.h) and returns its
status code; create functions return (status, handle).  Device memory and
streams come from the caller (PyTorch tensors' data_ptr() and
torch.cuda.Stream.cuda_stream work).  There is no fallback: if the compiled
library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_char_p, c_float, c_int32, c_size_t, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libllama_block.so")

LLAMA_OK = 0
LLAMA_ERR_INVALID_ARG = 1
LLAMA_ERR_SHAPE = 2
LLAMA_ERR_ALIGN = 3
LLAMA_ERR_RANGE = 4
LLAMA_ERR_UNSUPPORTED = 5
LLAMA_ERR_OOM = 6
LLAMA_ERR_CUDA = 7
LLAMA_ERR_DEVICE_TIMEOUT = 8

LLAMA_F32 = 0
LLAMA_BF16 = 1
LLAMA_ROPE_INTERLEAVED = 0
LLAMA_ROPE_HALVES = 1
LLAMA_DECODE_KERNELS = 0
LLAMA_DECODE_FUSED = 1

EPI_STORE = 0
EPI_RESIDUAL = 1
EPI_F32OUT = 2


class LlamaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        detail = f" [{llama_last_cuda_error()}]" if status == LLAMA_ERR_CUDA else ""
        super().__init__(f"{what}: {llama_status_string(status)} ({status}){detail}")


class llama_config(ctypes.Structure):
    _fields_ = [("d_model", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32), ("d_ff", c_int32),
                ("max_seq_len", c_int32), ("norm_eps", c_float), ("rope_theta", c_float), ("dtype", c_int32),
                ("rope_layout", c_int32), ("rope_scaling_factor", c_float), ("rope_low_freq_factor", c_float),
                ("rope_high_freq_factor", c_float), ("rope_original_max_pos", c_int32),
                ("n_experts", c_int32), ("top_k", c_int32), ("d_ff_shared", c_int32)]


WEIGHT_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
MOE_WEIGHT_FIELDS = ("router", "shared_gate", "shared_up", "shared_down")


class llama_block_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in WEIGHT_FIELDS + MOE_WEIGHT_FIELDS]


class llama_kv_cache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("max_batch", c_int32), ("max_seq_len", c_int32)]


_lib = None


def load() -> ctypes.CDLL:
    """Load the library (once).  Raises OSError when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError(f"{LIB_PATH} is missing: build it with decoder_block_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    st = c_int32
    sigs = {
        "llama_block_create": (st, [POINTER(llama_config), POINTER(llama_block_weights), c_int32, POINTER(c_void_p)]),
        "llama_block_forward": (st, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                     POINTER(llama_kv_cache), c_void_p]),
        "llama_block_forward_host": (st, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                          POINTER(llama_kv_cache), c_void_p]),
        "llama_block_destroy": (None, [c_void_p]),
        "llama_block_device_status": (st, [c_void_p]),
        "llama_block_set_decode_mode": (st, [c_void_p, c_int32]),
        "llama_stack_set_decode_mode": (st, [c_void_p, c_int32]),
        "llama_block_set_wait_budget": (st, [c_void_p, ctypes.c_int64]),
        "llama_stack_set_wait_budget": (st, [c_void_p, ctypes.c_int64]),
        "llama_stack_create": (st, [POINTER(llama_config), c_int32, c_int32, c_void_p, POINTER(llama_block_weights),
                                    c_void_p, c_void_p, c_int32, POINTER(c_void_p)]),
        "llama_stack_generate": (st, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                      POINTER(llama_kv_cache), c_void_p, c_void_p, c_void_p]),
        "llama_stack_forward": (st, [c_void_p, c_void_p, c_int32, c_int32, c_int32, POINTER(llama_kv_cache),
                                     c_void_p, c_void_p]),
        "llama_stack_destroy": (None, [c_void_p]),
        "llama_stack_device_status": (st, [c_void_p]),
        "llama_kv_cache_bytes": (c_size_t, [POINTER(llama_config), c_int32, c_int32]),
        "llama_block_profile_enable": (st, [c_void_p, c_int32]),
        "llama_block_profile_disable": (st, [c_void_p]),
        "llama_block_profile_read": (st, [c_void_p, POINTER(c_int32), POINTER(c_float)]),
        "llama_profile_step_name": (c_char_p, [c_int32]),
        "llama_ffn_hidden_dim": (c_int32, [c_int32, c_int32, c_float]),
        "llama_status_string": (c_char_p, [c_int32]),
        "llama_last_cuda_error": (c_char_p, []),
        "llama_block_moe_routing": (st, [c_void_p, c_void_p, c_void_p, c_void_p]),
        "llama_kernel_launch_count": (ctypes.c_ulonglong, []),
        "llama_op_rmsnorm": (st, [c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float, c_void_p]),
        "llama_op_linear": (st, [c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                                 c_void_p]),
        "llama_op_attention_workspace_bytes": (c_size_t, [c_int32, c_int32, c_int32, c_int32, c_int32, c_int32]),
        "llama_op_attention": (st, [c_int32, c_void_p, POINTER(llama_kv_cache), c_void_p, c_int32, c_int32, c_int32,
                                    c_int32, c_int32, c_int32, c_void_p, c_size_t, c_void_p]),
        "llama_op_rope_table": (st, [c_void_p, c_int32, c_int32, c_float, c_float, c_float, c_float, c_int32,
                                     c_void_p]),
        "llama_op_attention_decode_noalloc": (st, [c_void_p, POINTER(llama_kv_cache), c_void_p, c_int32, c_int32,
                                                   c_int32, c_int32, c_int32, c_void_p]),
        "llama_op_rope_kv_write": (st, [c_int32, c_void_p, c_void_p, POINTER(llama_kv_cache), c_void_p, c_int32,
                                        c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(x):
    """A raw pointer from an int, None, or anything with data_ptr()."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


# ---------------------------------------------------------------- structs ---

def make_config(d_model, n_heads, n_kv_heads, d_ff, max_seq_len, norm_eps, rope_theta, dtype,
                rope_layout=0, rope_scaling=None, n_experts=0, top_k=0, d_ff_shared=0) -> llama_config:
    """rope_scaling: None or a dict with factor, low_freq_factor, high_freq_factor, original_max_pos.
    n_experts > 0 makes the feed-forward a mixture of experts (d_ff is then each expert's width)."""
    sc = rope_scaling or {}
    return llama_config(d_model, n_heads, n_kv_heads, d_ff, max_seq_len, norm_eps, rope_theta, dtype, rope_layout,
                        float(sc.get("factor", 0.0)), float(sc.get("low_freq_factor", 0.0)),
                        float(sc.get("high_freq_factor", 0.0)), int(sc.get("original_max_pos", 0)),
                        n_experts, top_k, d_ff_shared)


def make_weights(w: dict) -> llama_block_weights:
    """Pointers of a weight dict (mixture-of-experts entries are optional)."""
    return llama_block_weights(*[_p(w[n]) for n in WEIGHT_FIELDS], *[_p(w.get(n)) for n in MOE_WEIGHT_FIELDS])


def make_kv_cache(k, v, max_batch, max_seq_len) -> llama_kv_cache:
    return llama_kv_cache(_p(k), _p(v), max_batch, max_seq_len)


# ------------------------------------------------------------ entry points ---

def llama_block_create(cfg: llama_config, weights: llama_block_weights, max_tokens: int):
    h = c_void_p()
    s = load().llama_block_create(byref(cfg), byref(weights), max_tokens, byref(h))
    return s, h.value


def llama_block_forward(blk, x, y, B, S, start_pos, kv: llama_kv_cache, stream=None) -> int:
    return load().llama_block_forward(blk, _p(x), _p(y), B, S, start_pos, byref(kv), _stream(stream))


def llama_block_forward_host(blk, x_host, y_host, B, S, start_pos, kv: llama_kv_cache, stream=None) -> int:
    return load().llama_block_forward_host(blk, _p(x_host), _p(y_host), B, S, start_pos, byref(kv), _stream(stream))


def llama_block_destroy(blk) -> None:
    load().llama_block_destroy(blk)


def llama_block_device_status(blk) -> int:
    return load().llama_block_device_status(blk)


def llama_block_set_decode_mode(blk, mode: int) -> int:
    return load().llama_block_set_decode_mode(blk, mode)


def llama_stack_set_decode_mode(stk, mode: int) -> int:
    return load().llama_stack_set_decode_mode(stk, mode)


def llama_block_set_wait_budget(blk, cycles: int) -> int:
    return load().llama_block_set_wait_budget(blk, cycles)


def llama_stack_set_wait_budget(stk, cycles: int) -> int:
    return load().llama_stack_set_wait_budget(stk, cycles)


def llama_stack_create(cfg: llama_config, n_layers, vocab, embed, layers, final_norm, lm_head, max_tokens):
    arr = (llama_block_weights * max(n_layers, 1))(*layers)
    h = c_void_p()
    s = load().llama_stack_create(byref(cfg), n_layers, vocab, _p(embed), arr, _p(final_norm), _p(lm_head),
                                  max_tokens, byref(h))
    return s, h.value


def llama_stack_forward(stk, tokens, B, S, start_pos, kv_list, logits, stream=None) -> int:
    arr = (llama_kv_cache * max(len(kv_list), 1))(*kv_list)
    return load().llama_stack_forward(stk, _p(tokens), B, S, start_pos, arr, _p(logits), _stream(stream))


def llama_stack_generate(stk, prompt, B, S_prompt, start_pos, n_new, kv_list, out_tokens, logits,
                         stream=None) -> int:
    arr = (llama_kv_cache * max(len(kv_list), 1))(*kv_list)
    return load().llama_stack_generate(stk, _p(prompt), B, S_prompt, start_pos, n_new, arr, _p(out_tokens),
                                       _p(logits), _stream(stream))


def llama_stack_destroy(stk) -> None:
    load().llama_stack_destroy(stk)


def llama_stack_device_status(stk) -> int:
    return load().llama_stack_device_status(stk)


LLAMA_PROFILE_STEPS = 8


def llama_block_profile_enable(blk, max_forwards) -> int:
    return load().llama_block_profile_enable(blk, max_forwards)


def llama_block_profile_disable(blk) -> int:
    return load().llama_block_profile_disable(blk)


def llama_block_profile_read(blk):
    """Returns (status, launches[8], total_ms[8])."""
    n = (c_int32 * LLAMA_PROFILE_STEPS)()
    ms = (c_float * LLAMA_PROFILE_STEPS)()
    s = load().llama_block_profile_read(blk, n, ms)
    return s, list(n), list(ms)


def llama_profile_step_name(step) -> str:
    return load().llama_profile_step_name(step).decode()


def llama_kv_cache_bytes(cfg: llama_config, max_batch, max_seq_len) -> int:
    return load().llama_kv_cache_bytes(byref(cfg), max_batch, max_seq_len)


def llama_ffn_hidden_dim(d_model, multiple_of, ffn_dim_multiplier) -> int:
    return load().llama_ffn_hidden_dim(d_model, multiple_of, ffn_dim_multiplier)


def llama_status_string(status) -> str:
    return load().llama_status_string(status).decode()


def llama_last_cuda_error() -> str:
    return load().llama_last_cuda_error().decode()


def llama_block_moe_routing(blk, ids, weights, stream=None) -> int:
    return load().llama_block_moe_routing(blk, _p(ids), _p(weights), _stream(stream))


def llama_kernel_launch_count() -> int:
    return int(load().llama_kernel_launch_count())


def llama_op_rmsnorm(dtype, x, g, out, T, d, eps, stream=None) -> int:
    return load().llama_op_rmsnorm(dtype, _p(x), _p(g), _p(out), T, d, eps, _stream(stream))


def llama_op_linear(dtype, A, W, R, C, M, N, K, epilogue, stream=None) -> int:
    return load().llama_op_linear(dtype, _p(A), _p(W), _p(R), _p(C), M, N, K, epilogue, _stream(stream))


def llama_op_attention_workspace_bytes(dtype, B, S, start_pos, H, D) -> int:
    return load().llama_op_attention_workspace_bytes(dtype, B, S, start_pos, H, D)


def llama_op_attention(dtype, q, kv: llama_kv_cache, o, B, S, start_pos, H, G, D, workspace=None, workspace_bytes=0,
                       stream=None) -> int:
    return load().llama_op_attention(dtype, _p(q), byref(kv), _p(o), B, S, start_pos, H, G, D, _p(workspace),
                                     workspace_bytes, _stream(stream))


def llama_op_rope_table(table, max_seq, D, theta, scaling=None, stream=None) -> int:
    sc = scaling or {}
    return load().llama_op_rope_table(_p(table), max_seq, D, theta, float(sc.get("factor", 0.0)),
                                      float(sc.get("low_freq_factor", 0.0)), float(sc.get("high_freq_factor", 0.0)),
                                      int(sc.get("original_max_pos", 0)), _stream(stream))


def llama_op_rope_kv_write(dtype, qkv, q_out, kv: llama_kv_cache, table, table_max_seq, B, S, start_pos, H, G, D,
                           layout=0, stream=None) -> int:
    return load().llama_op_rope_kv_write(dtype, _p(qkv), _p(q_out), byref(kv), _p(table), table_max_seq, B, S,
                                         start_pos, H, G, D, layout, _stream(stream))


LLAMA_NOALLOC_SCRATCH_BYTES = 32 << 20


def llama_op_attention_decode_noalloc(q, kv: llama_kv_cache, o, B, start_pos, H, G, D, stream=None) -> int:
    """Decode attention using the library's built-in scratch array (no device allocation)."""
    return load().llama_op_attention_decode_noalloc(_p(q), byref(kv), _p(o), B, start_pos, H, G, D, _stream(stream))


def check(status: int, what: str = "llama call") -> None:
    """Raise LlamaError for a non-OK status."""
    if status != LLAMA_OK:
        raise LlamaError(status, what)
