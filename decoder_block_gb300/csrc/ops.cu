// Per-step C entry points (llama_ops.h): validation + one kernel launch each.
#include "llama_ops.h"
#include "kernels.h"
#include "tc_kernels.h"

using namespace llama;

namespace {

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool device_ptr(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

llama_status check(const void *p) {
  if (p == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(p)) return LLAMA_ERR_ALIGN;
  return device_ptr(p) ? LLAMA_OK : LLAMA_ERR_INVALID_ARG;
}

llama_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return LLAMA_OK;
  note_cuda_error(e);
  return LLAMA_ERR_CUDA;
}

bool head_dim_ok(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }

}  // namespace

extern "C" {

llama_status llama_op_rmsnorm(int32_t dtype, const void *x, const void *g, void *out, int32_t T, int32_t d,
                              float eps, llama_stream stream) {
  if (dtype != LLAMA_F32 && dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (T < 0 || d <= 0 || !(eps >= 0.f)) return LLAMA_ERR_INVALID_ARG;
  if (d % (dtype == LLAMA_BF16 ? 8 : 4) != 0) return LLAMA_ERR_UNSUPPORTED;
  for (const void *p : {x, g, (const void *)out}) {
    llama_status s = check(p);
    if (s != LLAMA_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == LLAMA_BF16)
    return status_of(launch_rmsnorm<bf16>((const bf16 *)x, (const bf16 *)g, (bf16 *)out, T, d, eps, st));
  return status_of(launch_rmsnorm<float>((const float *)x, (const float *)g, (float *)out, T, d, eps, st));
}

llama_status llama_op_linear(int32_t dtype, const void *A, const void *W, const void *R, void *C, int32_t M,
                             int32_t N, int32_t K, int32_t epilogue, llama_stream stream) {
  if (dtype != LLAMA_F32 && dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  if (epilogue != EPI_STORE && epilogue != EPI_RESIDUAL && epilogue != EPI_F32OUT) return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  for (const void *p : {A, W, (const void *)C}) {
    llama_status s = check(p);
    if (s != LLAMA_OK) return s;
  }
  if (epilogue == EPI_RESIDUAL) {
    llama_status s = check(R);
    if (s != LLAMA_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == LLAMA_BF16)
    return status_of(
        launch_gemm_tc((const bf16 *)A, (const bf16 *)W, (const bf16 *)R, C, M, N, K, epilogue, nullptr, st));
  return status_of(
      launch_gemm_simt<float>((const float *)A, (const float *)W, nullptr, (const float *)R, C, M, N, K, epilogue, st));
}

size_t llama_op_attention_workspace_bytes(int32_t dtype, int32_t B, int32_t S, int32_t start_pos, int32_t H,
                                          int32_t D) {
  if (dtype != LLAMA_BF16 || S != 1 || B <= 0 || H <= 0 || start_pos < 0 || !head_dim_ok(D)) return 0;
  if (start_pos + 1 <= 256) return 0;  // a single chunk normalises in place
  return attn_decode_scratch_bytes(B, H, D, start_pos + 1);
}

llama_status llama_op_attention(int32_t dtype, const void *q, const llama_kv_cache *kv, void *o, int32_t B,
                                int32_t S, int32_t start_pos, int32_t H, int32_t G, int32_t D, void *workspace,
                                size_t workspace_bytes, llama_stream stream) {
  if (dtype != LLAMA_F32 && dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (kv == nullptr || B <= 0 || S <= 0 || start_pos < 0 || H <= 0 || G <= 0 || D <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (H % G != 0) return LLAMA_ERR_SHAPE;
  if (!head_dim_ok(D)) return LLAMA_ERR_UNSUPPORTED;
  if (B > kv->max_batch || (long long)start_pos + S > kv->max_seq_len) return LLAMA_ERR_RANGE;
  for (const void *p : {q, (const void *)kv->k, (const void *)kv->v, (const void *)o}) {
    llama_status s = check(p);
    if (s != LLAMA_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == LLAMA_BF16) {
    const size_t need = llama_op_attention_workspace_bytes(dtype, B, S, start_pos, H, D);
    if (need > 0) {
      if (workspace_bytes < need) return LLAMA_ERR_RANGE;
      llama_status s = check(workspace);
      if (s != LLAMA_OK) return s;
    }
    AttnScratch ws;
    ws.partial = need > 0 ? workspace : nullptr;
    ws.bytes = need > 0 ? workspace_bytes : 0;
    return status_of(launch_attention((const bf16 *)q, (const bf16 *)kv->k, (const bf16 *)kv->v, (bf16 *)o, B, S,
                                      start_pos, H, G, D, kv->max_seq_len, ws, nullptr, st));
  }
  return status_of(launch_attention_simt<float>((const float *)q, (const float *)kv->k, (const float *)kv->v,
                                                (float *)o, B, S, start_pos, H, G, D, kv->max_seq_len, st));
}

llama_status llama_op_rope_table(float *table, int32_t max_seq, int32_t D, float theta, float scaling_factor,
                                 float low_freq_factor, float high_freq_factor, int32_t original_max_pos,
                                 llama_stream stream) {
  if (max_seq <= 0 || D <= 0 || D % 2 != 0 || !(theta > 0.f)) return LLAMA_ERR_INVALID_ARG;
  RopeScaling sc;
  if (scaling_factor > 1.f) {
    if (!(low_freq_factor > 0.f && high_freq_factor > low_freq_factor && original_max_pos > 0))
      return LLAMA_ERR_INVALID_ARG;
    sc.factor = scaling_factor;
    sc.low = low_freq_factor;
    sc.high = high_freq_factor;
    sc.original_max_pos = original_max_pos;
  } else if (!(scaling_factor <= 1.f)) {
    return LLAMA_ERR_INVALID_ARG;
  }
  llama_status s = check(table);
  if (s != LLAMA_OK) return s;
  return status_of(launch_rope_table(reinterpret_cast<float2 *>(table), max_seq, D, (double)theta, sc,
                                     (cudaStream_t)stream));
}

llama_status llama_op_rope_kv_write(int32_t dtype, const void *qkv, void *q_out, const llama_kv_cache *kv,
                                    const float *table, int32_t table_max_seq, int32_t B, int32_t S,
                                    int32_t start_pos, int32_t H, int32_t G, int32_t D, int32_t layout,
                                    llama_stream stream) {
  if (dtype != LLAMA_F32 && dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (layout != LLAMA_ROPE_INTERLEAVED && layout != LLAMA_ROPE_HALVES) return LLAMA_ERR_INVALID_ARG;
  if (kv == nullptr || B <= 0 || S <= 0 || start_pos < 0 || H <= 0 || G <= 0 || D <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (H % G != 0) return LLAMA_ERR_SHAPE;
  if (!head_dim_ok(D)) return LLAMA_ERR_UNSUPPORTED;
  if (B > kv->max_batch || (long long)start_pos + S > kv->max_seq_len || (long long)start_pos + S > table_max_seq)
    return LLAMA_ERR_RANGE;
  for (const void *p : {qkv, (const void *)q_out, (const void *)kv->k, (const void *)kv->v, (const void *)table}) {
    llama_status s = check(p);
    if (s != LLAMA_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const float2 *t2 = reinterpret_cast<const float2 *>(table);
  if (dtype == LLAMA_BF16)
    return status_of(launch_rope_kv<bf16>((const bf16 *)qkv, (bf16 *)q_out, (bf16 *)kv->k, (bf16 *)kv->v, t2, B, S,
                                          start_pos, H, G, D, kv->max_seq_len, layout, st));
  return status_of(launch_rope_kv<float>((const float *)qkv, (float *)q_out, (float *)kv->k, (float *)kv->v, t2, B,
                                         S, start_pos, H, G, D, kv->max_seq_len, layout, st));
}

}  // extern "C"
