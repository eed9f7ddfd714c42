/*
 * llama_ops.h -- per-step entry points of the decoder block (same kernels the
 * block forward launches), for unit-level parity checks and for callers that
 * compose the steps themselves.  Conventions as in llama_block.h: device
 * pointers, 16-byte alignment, row-major, asynchronous on `stream`, errors
 * returned (nothing enqueued on error).  dtype is LLAMA_F32 or LLAMA_BF16.
 * These entry points allocate nothing and report device-side wait expiry only
 * through their return of later calls' CUDA errors (no status word).
 */
#ifndef LLAMA_OPS_H
#define LLAMA_OPS_H

#include "llama_block.h"

#ifdef __cplusplus
extern "C" {
#endif

/* RMSNorm of T rows of width d ("The Evolving Transformer 04 · LLaMA", §03):
 * out[t] = x[t] / sqrt(mean(x[t]^2) + eps) * g.  x, out: [T][d]; g: [d].
 * d must be a multiple of 8 (bf16) or 4 (fp32).  out may alias x. */
llama_status llama_op_rmsnorm(int32_t dtype, const void *x, const void *g, void *out, int32_t T, int32_t d,
                              float eps, llama_stream stream);

/* Linear layer without bias ("The Evolving Transformer 04 · LLaMA", §05: nn.Linear(bias=False)):
 *   epilogue 0: C = A W^T            C [M][N], dtype
 *   epilogue 1: C = R + A W^T        R, C [M][N], dtype (C may alias R)
 *   epilogue 2: C = A W^T            C [M][N], fp32
 * A: [M][K]; W: [N][K].  K must be a multiple of 8.  bf16 runs on the tcgen05
 * tensor cores with fp32 accumulation; fp32 runs on CUDA cores. */
llama_status llama_op_linear(int32_t dtype, const void *A, const void *W, const void *R, void *C, int32_t M,
                             int32_t N, int32_t K, int32_t epilogue, llama_stream stream);

/* Causal grouped-query attention over a KV cache ("The Evolving Transformer 04
 * · LLaMA", §05 GQA; "Full Llama 3 transformer block", How it works):
 * o[b][s][h] = sum_{j <= start_pos + s} softmax_j(q[b][s][h] . K[b][h / (H/G)][j] / sqrt(D)) V[b][h / (H/G)][j].
 * q, o: [B][S][H][D] (q already rotated); kv->k, kv->v: [max_batch][G][max_seq_len][D].
 * Requirements as for llama_block_forward; D in {16, 32, 64, 128}.
 * workspace: caller-owned device scratch of at least
 * llama_op_attention_workspace_bytes(dtype, B, S, start_pos, H, D) bytes
 * (the split-KV partials of the decode path); may be NULL when that is 0. */
size_t llama_op_attention_workspace_bytes(int32_t dtype, int32_t B, int32_t S, int32_t start_pos, int32_t H,
                                          int32_t D);
llama_status llama_op_attention(int32_t dtype, const void *q, const llama_kv_cache *kv, void *o, int32_t B,
                                int32_t S, int32_t start_pos, int32_t H, int32_t G, int32_t D, void *workspace,
                                size_t workspace_bytes, llama_stream stream);

/* RoPE cos/sin table: table[p][i] = {cos(p f_i), sin(p f_i)}, f_i = theta^(-2i/D),
 * p in [0, max_seq), i in [0, D/2), fp32 pairs computed in fp64 ("Mini Llama 2
 * Implementation", Rotary positional embeddings).  table: float[max_seq][D/2][2].
 * scaling_factor > 1 applies the Llama 3.1 stretch to f_i with low_freq_factor,
 * high_freq_factor and original_max_pos exactly as the llama_config fields of the
 * same names describe; scaling_factor <= 1 leaves f_i unscaled (the other three
 * are then ignored). */
llama_status llama_op_rope_table(float *table, int32_t max_seq, int32_t D, float theta, float scaling_factor,
                                 float low_freq_factor, float high_freq_factor, int32_t original_max_pos,
                                 llama_stream stream);

/* RoPE + KV-cache write: qkv [B*S][(H + 2G) D] holds, per token, q (H heads),
 * k (G heads), v (G heads).  Writes q rotated at position start_pos + s to
 * q_out [B*S][H][D], k rotated to kv->k[b][g][start_pos + s], v unrotated to
 * kv->v[b][g][start_pos + s]; nothing else in the cache changes.  layout
 * (llama_rope_layout) picks the pairs rotated together; the vectors keep their
 * natural component order in both layouts.
 * table from llama_op_rope_table with max_seq >= start_pos + S. */
llama_status llama_op_rope_kv_write(int32_t dtype, const void *qkv, void *q_out, const llama_kv_cache *kv,
                                    const float *table, int32_t table_max_seq, int32_t B, int32_t S,
                                    int32_t start_pos, int32_t H, int32_t G, int32_t D, int32_t layout,
                                    llama_stream stream);

/* Decode-step attention that allocates nothing.  The method's pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory when they run attention (a serving engine whose pool already owns
 * the device memory, an embedded runtime with a fixed budget, code that must
 * not synchronise the device the way cudaMalloc can).
 *
 * Computes the same as llama_op_attention with dtype LLAMA_BF16 and S = 1:
 * q, o: [B][H][D] bf16, kv: bf16 [max_batch][G][max_seq_len][D], keys
 * 0 .. start_pos visible.  The split-KV partial results live in one array of
 * LLAMA_NOALLOC_SCRATCH_BYTES that is part of the library image on every GPU
 * that loads it, held until the process exits; no cudaMalloc / cudaFree or
 * allocating library routine is called.
 *   - Limit: one sequence's partials, H * ceil((start_pos + 1) / 256) *
 *     (D + 2) * 4 bytes, must fit in LLAMA_NOALLOC_SCRATCH_BYTES, else
 *     LLAMA_ERR_RANGE (nothing runs); a single chunk (start_pos < 256) needs
 *     none.  Batches whose partials do not fit run in groups of sequences, one
 *     group after another on the stream, each reusing the array.  With
 *     H = 32 and D = 128 a sequence needs 16,640 bytes per 256 positions:
 *     32 MiB holds one sequence of up to 516,096 cached positions, and B = 64
 *     sequences of 4096 positions in one group.
 *   - D in {64, 128}, n_heads / n_kv_heads <= 8 (LLAMA_ERR_UNSUPPORTED otherwise).
 *   - The first call on a device looks up the array's device address (a
 *     one-time set-up per CUDA context, done with that device current, and
 *     done again after the device's context was reset); make that first call
 *     before any stream capture.
 *   - All calls share the array and every call overwrites the partials it
 *     reads, so nothing needs clearing; calls that may run at the same time on
 *     the GPU (unordered streams) race on the array and must be avoided.
 *   - The kernel's bounded waits (2 s, never reached in normal operation)
 *     have no status word to report to here: if one ran out, the call still
 *     returns LLAMA_OK and o is undefined. */
#define LLAMA_NOALLOC_SCRATCH_BYTES (32u << 20)
llama_status llama_op_attention_decode_noalloc(const void *q, const llama_kv_cache *kv, void *o, int32_t B,
                                               int32_t start_pos, int32_t H, int32_t G, int32_t D,
                                               llama_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* LLAMA_OPS_H */
