// Launcher of the tensor-core decode attention (kernel body: decode_tc_body.cuh).
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_tc_body.cuh"

namespace llama {
namespace {

template <int RN>
__global__ void __launch_bounds__(DT_THREADS, 1)
    attn_decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ DtArgs a) {
  attn_decode_tc_run<RN>(&tmQ, &tmK, &tmV, a, PhaseSync{});
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool encode(CUtensorMap *map, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides,
            const uint32_t *box) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gd[4];
  cuuint64_t gs[3];
  cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), gd, gs, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_decode_tc_supported(int H, int G, int D) { return D == DT_D && H % G == 0 && H / G <= DT_N; }

size_t attn_decode_tc_scratch_bytes(int B, int H, int kv_len) {
  const int n_split = (kv_len + DT_CHUNK - 1) / DT_CHUNK;
  return n_split > 1 ? (size_t)B * H * n_split * (DT_D + 2) * sizeof(float) : 0;
}

cudaError_t attn_decode_tc_prepare(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos,
                                   int H, int G, int cache_seq, const AttnScratch &scratch, int *status,
                                   CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv, DtArgs *out) {
  if (B <= 0 || G <= 0 || !attn_decode_tc_supported(H, G, DT_D)) return cudaErrorInvalidValue;
  DtArgs a;
  a.B = B;
  a.H = H;
  a.G = G;
  a.r = H / G;
  a.kv_len = start_pos + 1;
  a.n_split = (a.kv_len + DT_CHUNK - 1) / DT_CHUNK;
  a.n_items = B * G * a.n_split;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)DT_D);
  a.status = status;
  a.o = o;
  a.part = reinterpret_cast<float *>(scratch.partial);
  a.items = scratch.item_counters;
  if (a.n_split > 1 && (scratch.partial == nullptr ||
                        scratch.bytes < attn_decode_tc_scratch_bytes(B, H, a.kv_len)))
    return cudaErrorInvalidValue;
  const uint64_t qd[2] = {(uint64_t)DT_D, (uint64_t)B * H};
  const uint64_t qs[1] = {(uint64_t)DT_D * 2};
  const uint32_t qb[2] = {64, DT_N};
  const uint64_t kd[4] = {(uint64_t)DT_D, (uint64_t)a.kv_len, (uint64_t)G, (uint64_t)B};
  const uint64_t ks[3] = {(uint64_t)DT_D * 2, (uint64_t)cache_seq * DT_D * 2, (uint64_t)G * cache_seq * DT_D * 2};
  const uint32_t kb[4] = {64, DT_TILE, 1, 1};
  if (!encode(mq, q, 2, qd, qs, qb) || !encode(mk, kc, 4, kd, ks, kb) || !encode(mv, vc, 4, kd, ks, kb))
    return cudaErrorInvalidValue;
  *out = a;
  return cudaSuccess;
}

cudaError_t launch_attn_decode_tc(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos,
                                  int H, int G, int cache_seq, const AttnScratch &scratch, int *status,
                                  cudaStream_t st) {
  static PerContextOnce attr;
  const cudaError_t attr_err = attr.run([] {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DtLayout::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_decode_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DtLayout::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_decode_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DtLayout::BYTES);
    return e;
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap mq, mk, mv;
  DtArgs a;
  cudaError_t e = attn_decode_tc_prepare(q, kc, vc, o, B, start_pos, H, G, cache_seq, scratch, status, &mq, &mk, &mv,
                                         &a);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.n_items < sms ? a.n_items : sms;
  count_launch();
  auto kernel = a.r <= 4 ? attn_decode_tc_kernel<4> : (a.r <= 8 ? attn_decode_tc_kernel<8> : attn_decode_tc_kernel<16>);
  e = launch_pdl(kernel, dim3(grid), dim3(DT_THREADS), DtLayout::BYTES, st, mq, mk, mv, a);
  if (e != cudaSuccess || a.n_split == 1) return e;
  return launch_decode_combine(a.part, o, B * H, DT_D, a.n_split, st);
}

}  // namespace llama
