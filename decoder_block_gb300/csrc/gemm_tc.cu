// Persistent, warp-specialised tcgen05 GEMM for the four dense projections of
// the block (QKV, O, gate/up, down) and the LM head:  C = epi(A W^T), with A
// [M,K] activations and W [N,K] nn.Linear weights, both bf16 and K-major.
//
// Per CTA (one per SM, 192 threads):
//   warp 0      TMA producer: 128x64 A box + 256x64 W box per stage, 128-byte
//               swizzle, STAGES-deep ring of shared-memory buffers;
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma (M=128, N=256,
//               K=16) from one thread into one of two 256-column fp32
//               accumulators, commits stage releases and accumulator-ready;
//   warps 2..5  epilogue: tcgen05.ld the accumulator rows of their TMEM lane
//               quarter, apply the fused epilogue (store / + residual /
//               SiLU(gate) * up / fp32 out) and store to global memory, then
//               hand the accumulator back -- overlapping the next tile's K loop.
// Every mbarrier wait is bounded (clock budget); on expiry the kernel records a
// status code, drains in-flight copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int GROUP_M = 16;

struct GemmArgs {
  const bf16 *R;
  void *C;
  int M, N, K;
  int *status;
};

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int &mt, int &nt) {
  const int per_group = GROUP_M * n_tiles;
  const int g = tile / per_group;
  const int first = g * GROUP_M;
  const int gm = min(m_tiles - first, GROUP_M);
  const int local = tile % per_group;
  mt = first + local % gm;
  nt = local / gm;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

template <int EPI>
__device__ __forceinline__ void epilogue_chunk16(const float (&v)[16], const GemmArgs &a, int m, int n) {
  // v holds columns n .. n+15 of row m (EPI_STORE / EPI_RESIDUAL / EPI_F32OUT).
  if (m >= a.M || n >= a.N) return;
  const size_t base = (size_t)m * a.N + n;
  if constexpr (EPI == EPI_F32OUT) {
    float *c = reinterpret_cast<float *>(a.C) + base;
    if (n + 16 <= a.N && (a.N & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4 *>(c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (n + i < a.N) c[i] = v[i];
    }
  } else {
    bf16 *c = reinterpret_cast<bf16 *>(a.C) + base;
    float w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = v[i];
    const bool vec = n + 16 <= a.N && (a.N & 7) == 0;
    if constexpr (EPI == EPI_RESIDUAL) {
      const bf16 *r = a.R + base;
      if (vec) {
        uint4 r0 = *reinterpret_cast<const uint4 *>(r), r1 = *reinterpret_cast<const uint4 *>(r + 8);
        const bf16 *p0 = reinterpret_cast<const bf16 *>(&r0), *p1 = reinterpret_cast<const bf16 *>(&r1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          w[i] += __bfloat162float(p0[i]);
          w[i + 8] += __bfloat162float(p1[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (n + i < a.N) w[i] += __bfloat162float(r[i]);
      }
    }
    if (vec) {
      uint4 o0 = make_uint4(pack_bf16(w[0], w[1]), pack_bf16(w[2], w[3]), pack_bf16(w[4], w[5]), pack_bf16(w[6], w[7]));
      uint4 o1 = make_uint4(pack_bf16(w[8], w[9]), pack_bf16(w[10], w[11]), pack_bf16(w[12], w[13]),
                            pack_bf16(w[14], w[15]));
      *reinterpret_cast<uint4 *>(c) = o0;
      *reinterpret_cast<uint4 *>(c + 8) = o1;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (n + i < a.N) c[i] = __float2bfloat16_rn(w[i]);
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t smem0 = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t fin_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (args.M + BM - 1) / BM, n_tiles = (args.N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int k_steps = (args.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), 128);
    }
    ptx::mbar_init(fin_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, m_tiles, n_tiles, mt, nt);
        for (int k = 0; k < k_steps; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1, abort_flag, args.status, DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem0 + s * STAGE_BYTES, sb = sa + A_BYTES;
          ptx::mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmA, k * BK, mt * BM, full_bar(s));
          ptx::tma_load_2d(sb, &tmB, k * BK, nt * BN, full_bar(s));
          ++it;
        }
      }
      // Every issued copy must have landed before the CTA can exit.
      for (int j = it - STAGES < 0 ? 0 : it - STAGES; j < it; ++j) {
        int dummy = 0;
        ptx::mbar_wait(full_bar(j % STAGES), (j / STAGES) & 1, &dummy, args.status, DEV_TIMEOUT_PRODUCER);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tcount) {
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!ptx::mbar_wait(tempty_bar(acc), aph ^ 1, abort_flag, args.status, DEV_TIMEOUT_MMA)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int k = 0; k < k_steps; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!ptx::mbar_wait(full_bar(s), ph, abort_flag, args.status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = smem0 + s * STAGE_BYTES, sb = sa + A_BYTES;
          const uint64_t adesc = ptx::smem_desc_sw128(sa), bdesc = ptx::smem_desc_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16_ss(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                             (k | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(empty_bar(s));
          ++it;
        }
        if (ok) ptx::mma_commit(tfull_bar(acc));
      }
      // Wait until every issued MMA has finished before TMEM / smem go away.
      ptx::mma_commit(fin_bar);
      int dummy = 0;
      ptx::mbar_wait(fin_bar, 0, &dummy, args.status, DEV_TIMEOUT_MMA);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
      int mt, nt;
      tile_coords(tile, m_tiles, n_tiles, mt, nt);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      bool ok = ptx::mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, DEV_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      const int m = mt * BM + row;
      if constexpr (EPI == EPI_SWIGLU) {
        const int nout = args.N / 2;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float gu[32];  // gate in columns c .. c+15, up in c+16 .. c+31
          ptx::tmem_ld32(trow + c, gu);
          const float *g = gu;
          const float *u = gu + 16;
          const int f = (nt * BN + c) / 2;
          if (m < args.M && f < nout) {
            bf16 *dst = reinterpret_cast<bf16 *>(args.C) + (size_t)m * nout + f;
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = pack_bf16(silu_f32(g[2 * i]) * u[2 * i], silu_f32(g[2 * i + 1]) * u[2 * i + 1]);
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float v[16];
          ptx::tmem_ld16(trow + c, v);
          ptx::tmem_ld_wait();
          epilogue_chunk16<EPI>(v, args, m, nt * BN + c);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(acc));
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows, 64], 128-byte swizzle.
bool make_map_2d(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int EPI>
cudaError_t launch_epi(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &args, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int tiles = ((args.M + BM - 1) / BM) * ((args.N + BN - 1) / BN);
  const int grid = tiles < sm_count() ? tiles : sm_count();
  gemm_tc_kernel<EPI><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ma, mb, args);
  return cudaGetLastError();
}

__global__ void interleave_rows_kernel(const uint4 *__restrict__ gate, const uint4 *__restrict__ up,
                                       uint4 *__restrict__ out, int F, int vec_per_row) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t total = (size_t)2 * F * vec_per_row;
  if (idx >= total) return;
  const int orow = (int)(idx / vec_per_row), c = (int)(idx % vec_per_row);
  const int j = orow / 32, i = orow % 32;
  const uint4 *src = i < 16 ? gate : up;
  const int srow = 16 * j + (i & 15);
  out[idx] = src[(size_t)srow * vec_per_row + c];
}

}  // namespace

cudaError_t launch_gemm_tc(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                           int *status, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (K <= 0 || (K & 7) != 0) return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && (N & 31) != 0) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  if (!make_map_2d(&ma, A, (uint64_t)M, (uint64_t)K, BM) || !make_map_2d(&mb, W, (uint64_t)N, (uint64_t)K, BN))
    return cudaErrorInvalidValue;
  GemmArgs args{R, C, M, N, K, status};
  switch (epi) {
    case EPI_STORE: return launch_epi<EPI_STORE>(ma, mb, args, st);
    case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL>(ma, mb, args, st);
    case EPI_F32OUT: return launch_epi<EPI_F32OUT>(ma, mb, args, st);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(ma, mb, args, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_interleave_rows(const bf16 *gate, const bf16 *up, bf16 *out, int F, int d, cudaStream_t st) {
  if ((F & 15) != 0 || (d & 7) != 0) return cudaErrorInvalidValue;
  const int vpr = d / 8;
  const size_t total = (size_t)2 * F * vpr;
  interleave_rows_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const uint4 *>(gate), reinterpret_cast<const uint4 *>(up), reinterpret_cast<uint4 *>(out), F,
      vpr);
  return cudaGetLastError();
}

}  // namespace llama
