// Internal launch wrappers shared by the runtime (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace llama {

enum Epilogue : int {
  EPI_STORE = 0,     // C = A W^T                 (C in the input dtype)
  EPI_RESIDUAL = 1,  // C = R + A W^T             (R, C in the input dtype)
  EPI_F32OUT = 2,    // C = A W^T, C fp32
  EPI_SWIGLU = 3,    // C = SiLU(A W1^T) * (A W3^T)
  // RMSNorm fused into the consuming GEMM (gain folded into W at create time):
  // row m of the accumulator is scaled by rsqrt(ss[m] / d + eps).
  EPI_STORE_ROWSCALE = 4,   // C = r_m (A W^T)
  EPI_SWIGLU_ROWSCALE = 5,  // C = SiLU(r_m A W1^T) * (r_m A W3^T)
  // residual add that also accumulates ss_out[m] += sum_n C[m,n]^2 of the stored bf16 C
  EPI_RESIDUAL_SQSUM = 6,
  // QKV projection with the attention RMSNorm row scale, RoPE on the q and k
  // columns and the scatter of rotated q into q_out and of k / v into the cache
  EPI_QKV_ROPE = 7,
  EPI_F32OUT_ROWSCALE = 8,  // C fp32 = r_m (A W^T)  (mixture-of-experts router logits)
};

// ss[t] = sum_j x[t][j]^2 (fp32) for rows of width d; zero_out[t] = 0 when not null.
cudaError_t launch_row_sqsum(const bf16 *x, float *ss, float *zero_out, int rows, int d, cudaStream_t st,
                             float *zero_out2 = nullptr);

// W[n][k] <- bf16(W[n][k] * g[k]) in place (fold an RMSNorm gain into a weight).
cudaError_t launch_scale_columns(bf16 *W, const bf16 *g, int rows, int cols, cudaStream_t st);

// RMSNorm of `rows` rows of width d (d % (16 / sizeof(T)) == 0).
template <typename T>
cudaError_t launch_rmsnorm(const T *x, const T *g, T *out, int rows, int d, float eps, cudaStream_t st);

// Portable tiled GEMM with fp32 accumulation: C[M,N] = epi(A[M,K] W[N,K]^T).
// W3 is only read by EPI_SWIGLU.
template <typename T>
cudaError_t launch_gemm_simt(const T *A, const T *W, const T *W3, const T *R, void *C, int M, int N, int K,
                             int epi, cudaStream_t st);

// Llama 3.1 RoPE frequency stretch (factor <= 1: none); see llama_config.
struct RopeScaling {
  double factor = 0.0, low = 0.0, high = 0.0, original_max_pos = 0.0;
};

// cos/sin table [max_seq][D/2] (float2 = {cos, sin}) of p * f_i with
// f_i = theta^(-2i/D), stretched when sc.factor > 1; computed in fp64.
cudaError_t launch_rope_table(float2 *table, int max_seq, int D, double theta, const RopeScaling &sc,
                              cudaStream_t st);
// The same values grouped for the GEMM epilogue: [D/4][max_seq] float4 =
// {cos_2g, sin_2g, cos_2g+1, sin_2g+1} at (g, p), so that the 32 rows (consecutive
// positions) of a warp read one contiguous 512-byte run per pair group.
cudaError_t launch_rope_table_grouped(float2 *table, int max_seq, int D, double theta, const RopeScaling &sc,
                                      cudaStream_t st);

// RoPE on q and k of qkv [T][(H + 2G) D] and the KV-cache write.
//   q_out [T][H D] (rotated q); kc/vc [cache_batch][G][cache_seq][D].
// halves = 0: pairs (2i, 2i+1); 1: pairs (i, i + D/2); natural component order in and out.
template <typename T>
cudaError_t launch_rope_kv(const T *qkv, T *q_out, T *kc, T *vc, const float2 *table, int B, int S,
                           int start_pos, int H, int G, int D, int cache_seq, int halves, cudaStream_t st);

// Reference causal GQA attention: one warp per (token, query head), online softmax in fp32.
template <typename T>
cudaError_t launch_attention_simt(const T *q, const T *kc, const T *vc, T *o, int B, int S, int start_pos,
                                  int H, int G, int D, int cache_seq, cudaStream_t st);

// x[t] = E[tokens[t]]; an out-of-range id writes zeros and sets the status word.
template <typename T>
cudaError_t launch_embed(const int32_t *tokens, const T *E, T *x, int ntok, int d, int vocab, int *status,
                         cudaStream_t st);

// Mixture-of-experts routing and data movement (moe.cu).  E <= 256, k <= min(E, 32).
bool moe_supported(int E, int k);
// ids / wts [T][k]: the k largest logits of row t (logits [T][ld], fp32) and a
// softmax over them; counts[e] += number of choices of e (counts zero before).
cudaError_t launch_moe_topk(const float *logits, int ld, int T, int E, int k, int *ids, float *wts, int *counts,
                            cudaStream_t st);
// offsets [E + 1] = exclusive prefix sums of counts; counts and fill left zero.
cudaError_t launch_moe_offsets(int *counts, int *offsets, int *fill, int E, cudaStream_t st);
// For each (t, j): pos[t][j] = a free row of expert ids[t][j]'s range, and that
// row of xin = bf16(h[t] * rsqrt(ss[t] / d + eps) * g).
cudaError_t launch_moe_dispatch(const bf16 *h, const float *ss, const bf16 *g, float eps, int T, int d, int k,
                                const int *ids, const int *offsets, int *fill, int *pos, bf16 *xin, cudaStream_t st);
// y[t] = base[t] + sum_j wts[t][j] * ye[pos[t][j]] (rows of width d).
cudaError_t launch_moe_combine(const bf16 *base, const bf16 *ye, const int *pos, const float *wts, int T, int d,
                               int k, bf16 *y, cudaStream_t st);

// Greedy pick: out[r * out_stride] (and next[r], when not null) = arg-max of
// logits row r [rows][vocab] fp32, lowest id among equal maxima.
cudaError_t launch_argmax_rows(const float *logits, int rows, int vocab, int32_t *out, int out_stride, int32_t *next,
                               cudaStream_t st);

// out[b] = x[b][S - 1] (rows of width d; d % (16 / sizeof(T)) == 0).
template <typename T>
cudaError_t launch_gather_last_rows(const T *x, T *out, int B, int S, int d, cudaStream_t st);

}  // namespace llama
