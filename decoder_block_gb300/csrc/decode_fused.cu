// The decode step of a dense bf16 block as ONE kernel.
// "Full Llama 3 transformer block", How it works (one new token per sequence
// attends to the cached keys 0 .. start_pos); "The Evolving Transformer 04 ·
// LLaMA", §06 Block (pre-norm residual block).
//
// A decode step (S = 1, a few dozen tokens) is a chain of seven short,
// bandwidth-bound kernels; between two of them the GPU drains one kernel's
// last CTAs and fills the next one's pipelines.  Here the chain runs as phases
// of one cooperative kernel (one CTA of 192 threads per SM, all resident), with
// a grid-wide arrival counter between phases (phase_sync.cuh):
//   0  attention-norm statistics  sum(x^2) per row; sum(h^2) zeroed
//   1  QKV GEMM + RMSNorm row scale + RoPE + K/V cache write   (gemm_tc_body.cuh)
//   2  decode attention, split over 512-key chunks              (decode_tc_body.cuh)
//   3  merge of the chunk partials (one warp per (b, h) row)
//   4  O GEMM + residual + sum(h^2)
//   5  gate/up GEMM + ffn-norm row scale + SwiGLU
//   6  down GEMM + residual
// Each phase is the same device code as the corresponding kernel of the
// multi-kernel path, with the same tile plans, so both paths compute the same
// values (up to the order of fp32 reductions).  A CTA that has finished its
// part of a phase prepares the next one while the others finish: it may ask L2
// for the data of its next work unit (see the cross-phase prefetch below),
// then initialises the barriers and requests its first weight tiles into
// shared memory before it waits at the phase barrier.
// Every wait is bounded: a phase barrier that is not reached within the clock
// budget records DEV_TIMEOUT_PHASE in the status word and sets an abort word
// that makes every later wait give up at once.
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_tc_body.cuh"
#include "gemm_tc_body.cuh"

namespace llama {
namespace {

constexpr int FUSED_THREADS = 192;
static_assert(FUSED_THREADS == NUM_THREADS && FUSED_THREADS == DT_THREADS, "phases share one CTA shape");
constexpr uint32_t FUSED_TMEM_COLS = 512;  // the widest phase: two 256-column GEMM accumulators

constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int FUSED_SMEM = cmax(cmax(cmax(GemmCfg<256>::SMEM_BYTES, GemmCfg<192>::SMEM_BYTES),
                                     cmax(GemmCfg<128>::SMEM_BYTES, GemmCfg<64>::SMEM_BYTES)),
                                DtLayout::BYTES);

struct FusedMaps {
  CUtensorMap qkv_a, qkv_w, o_a, o_w, gu_a, gu_w, dn_a, dn_w, q, k, v;
};

struct FusedArgs {
  GemmArgs qkv, o, gu, dn;
  int bn_qkv, bn_o, bn_gu, bn_dn;
  DtArgs attn;
  const bf16 *x;   // [rows][d]
  float *ss_x;     // sum(x^2) per row (written by phase 0)
  float *ss_h;     // sum(h^2) per row (zeroed by phase 0, accumulated by phase 4)
  int rows, d;
  unsigned *sync;  // [0] phase arrivals, [1] abort word; zero at launch
};

// Phase 0: one row per CTA (rows beyond the grid loop); fp32 sum of squares.
__device__ __forceinline__ void rowsq_phase(const FusedArgs &a) {
  __shared__ float red[FUSED_THREADS / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const bf16 *xr = a.x + (size_t)row * a.d;
    float acc = 0.f;
    for (int i = threadIdx.x; i < a.d / 8; i += FUSED_THREADS) {
      Vec16<bf16> v = load16(xr + (size_t)i * 8);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float f = v.get(k);
        acc = fmaf(f, f, acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.f;
      for (int w = 0; w < FUSED_THREADS / 32; ++w) s += red[w];
      a.ss_x[row] = s;
      a.ss_h[row] = 0.f;
    }
    __syncthreads();
  }
}

template <int EPI>
__device__ __forceinline__ void gemm_phase(const CUtensorMap *ta, const CUtensorMap *tw, const GemmArgs &args, int bn,
                                        const PhaseSync s) {
  switch (bn) {
    case 256: gemm_tc_run<EPI, 256, false>(ta, tw, args, s); break;
    case 192: gemm_tc_run<EPI, 192, false>(ta, tw, args, s); break;
    case 128: gemm_tc_run<EPI, 128, false>(ta, tw, args, s); break;
    default: gemm_tc_run<EPI, 64, false>(ta, tw, args, s); break;
  }
}

__device__ __noinline__ void attn_phase(const FusedMaps &m, const DtArgs &a, const PhaseSync s) {
  if (a.r <= 4)
    attn_decode_tc_run<4>(&m.q, &m.k, &m.v, a, s);
  else if (a.r <= 8)
    attn_decode_tc_run<8>(&m.q, &m.k, &m.v, a, s);
  else
    attn_decode_tc_run<16>(&m.q, &m.k, &m.v, a, s);
}

// Phase 3: merge of the chunk partials, one warp per (b, h) row (the same
// merge as decode_combine.cuh).  Lane l owns d = 2l, 2l + 1, 64 + 2l, 65 + 2l;
// the chunks' (m, l) pairs are read 32 at a time, one per lane, and shared by
// shuffles, so every load of a row is independent of the others.
__device__ __noinline__ void combine_phase(const DtArgs &a, const PhaseSync s) {
  if (a.n_split <= 1) return;  // the attention phase wrote o itself
  __shared__ int ready;
  if (threadIdx.x == 0) ready = phase_wait(s, a.status) ? 1 : 0;
  __syncthreads();
  if (!ready) return;
  constexpr int W = DT_D + 2;  // floats per chunk partial: o[D], m, l
  const int lane = threadIdx.x & 31;
  const int warps = FUSED_THREADS / 32;
  const int BH = a.B * a.H;
  for (int bh = blockIdx.x * warps + (threadIdx.x >> 5); bh < BH; bh += gridDim.x * warps) {
    const float *p = a.part + (size_t)bh * a.n_split * W;
    float m = -INFINITY;
    for (int c = lane; c < a.n_split; c += 32) m = fmaxf(m, p[c * W + DT_D]);
    m = warp_max(m);
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, lpart = 0.f;
    for (int c0 = 0; c0 < a.n_split; c0 += 32) {
      float f = 0.f;
      if (c0 + lane < a.n_split) {
        const float mc = p[(c0 + lane) * W + DT_D];
        f = mc == -INFINITY ? 0.f : ptx::ex2_approx(mc - m);
        lpart = fmaf(f, p[(c0 + lane) * W + DT_D + 1], lpart);
      }
      const int cnt = min(32, a.n_split - c0);
#pragma unroll 8
      for (int j = 0; j < cnt; ++j) {
        const float fj = __shfl_sync(0xffffffffu, f, j);
        const float *oc = p + (c0 + j) * W;  // 8-byte aligned: W * 4 = 520 bytes per chunk
        const float2 u = *reinterpret_cast<const float2 *>(oc + 2 * lane);
        const float2 v = *reinterpret_cast<const float2 *>(oc + 64 + 2 * lane);
        acc[0] = fmaf(fj, u.x, acc[0]);
        acc[1] = fmaf(fj, u.y, acc[1]);
        acc[2] = fmaf(fj, v.x, acc[2]);
        acc[3] = fmaf(fj, v.y, acc[3]);
      }
    }
    const float inv = 1.f / warp_sum(lpart);
    bf16 *o = a.o + (size_t)bh * DT_D;
    *reinterpret_cast<__nv_bfloat162 *>(o + 2 * lane) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    *reinterpret_cast<__nv_bfloat162 *>(o + 64 + 2 * lane) = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  }
}

// Cross-phase prefetch.  A CTA that has finished its part of a phase asks L2
// for the data its first work unit of the next phase streams and that the
// phase in between does not write: the cached K/V tiles of its first attention
// item (after the QKV phase), the first weight boxes of its gate/up unit
// (after the O phase, whose split-K finishing warps leave the memory mostly
// idle).  The next phase's own TMA loads then hit L2.  Nothing waits on a
// prefetch.  (Measured on the Llama-3-8B decode step: requesting the QKV
// weights before the row statistics delayed those, and the O and down weights
// gained nothing; those are not requested.)
// Weight boxes of this CTA's first unit of a GEMM phase, at most max_steps K steps.
__device__ __forceinline__ void prefetch_gemm_w(const CUtensorMap *tw, const GemmArgs &args, int bn, int max_steps) {
  if (threadIdx.x != 0) return;
  const int tiles = ((args.M + BM - 1) / BM) * ((args.N + bn - 1) / bn);
  const int units = args.split_tiles * args.splits + tiles - args.split_tiles;
  if ((int)blockIdx.x >= units) return;
  int a_row, w_row, nt, k0, k1, slot;
  dense_unit(args, bn, blockIdx.x, a_row, w_row, nt, k0, k1, slot);
  const int kend = min(k1, k0 + max_steps);
  for (int k = k0; k < kend; ++k) ptx::tma_prefetch_l2_2d(tw, k * BK, w_row);
}

// K and V tiles of this CTA's first attention item (b, g, chunk).  The one
// tile that the QKV phase writes into (position start_pos) may be requested
// while it is being written: L2 is where both meet, so the later load reads
// the written values either way.
__device__ __forceinline__ void prefetch_attn_kv(const FusedMaps &m, const DtArgs &a) {
  if (threadIdx.x != 0 || (int)blockIdx.x >= a.n_items) return;
  const int it = blockIdx.x;
  const int bg = it / a.n_split;
  const int b = bg / a.G, g = bg % a.G;
  const int k0 = (it % a.n_split) * DT_CHUNK;
  const int k1 = min(a.kv_len, k0 + DT_CHUNK);
  for (int key = k0; key < k1; key += DT_TILE)
    for (int at = 0; at < 2; ++at) {
      ptx::tma_prefetch_l2_4d(&m.k, at * 64, key, g, b);
      ptx::tma_prefetch_l2_4d(&m.v, at * 64, key, g, b);
    }
}

// K steps of a GEMM unit's weights requested ahead: about 64 MB over all CTAs
// (half of L2), so that the prefetched boxes are still there when used.
__device__ __forceinline__ int prefetch_budget(const GemmArgs &args, int bn) {
  const int tiles = ((args.M + BM - 1) / BM) * ((args.N + bn - 1) / bn);
  const int units = args.split_tiles * args.splits + tiles - args.split_tiles;
  const long long per_step = (long long)min(units, (int)gridDim.x) * bn * BK * 2;
  return (int)max(1LL, (64LL << 20) / per_step);
}

__global__ void __launch_bounds__(FUSED_THREADS, 1)
    decode_block_fused_kernel(const __grid_constant__ FusedMaps m, const __grid_constant__ FusedArgs a) {
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), FUSED_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  PhaseSync s;
  s.arrivals = a.sync;
  s.tmem = tmem_slot;
  const unsigned grid = gridDim.x;

  rowsq_phase(a);  // x was written before the launch: no wait
  phase_arrive(s);
  s.target = 1 * grid;
  gemm_phase<EPI_QKV_ROPE>(&m.qkv_a, &m.qkv_w, a.qkv, a.bn_qkv, s);
  prefetch_attn_kv(m, a.attn);
  phase_arrive(s);
  s.target = 2 * grid;
  attn_phase(m, a.attn, s);
  phase_arrive(s);
  s.target = 3 * grid;
  combine_phase(a.attn, s);
  phase_arrive(s);
  s.target = 4 * grid;
  gemm_phase<EPI_RESIDUAL_SQSUM>(&m.o_a, &m.o_w, a.o, a.bn_o, s);
  prefetch_gemm_w(&m.gu_w, a.gu, a.bn_gu, prefetch_budget(a.gu, a.bn_gu));
  phase_arrive(s);
  s.target = 5 * grid;
  gemm_phase<EPI_SWIGLU_ROWSCALE>(&m.gu_a, &m.gu_w, a.gu, a.bn_gu, s);
  phase_arrive(s);
  s.target = 6 * grid;
  gemm_phase<EPI_RESIDUAL>(&m.dn_a, &m.dn_w, a.dn, a.bn_dn, s);

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_slot, FUSED_TMEM_COLS);
  }
}

int fused_grid() {
  static PerContextOnce attr;
  if (attr.run([] {
        return cudaFuncSetAttribute(decode_block_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    FUSED_SMEM);
      }) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  static std::once_flag once;
  static int grid = 0;
  std::call_once(once, [] {
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_block_fused_kernel, FUSED_THREADS,
                                                      FUSED_SMEM) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    if (coop && per_sm >= 1) grid = sms;  // one CTA per SM, every CTA resident
  });
  return grid;
}

}  // namespace

bool decode_fused_available() { return fused_grid() > 0; }

cudaError_t launch_decode_block_fused(const DecodeFusedParams &p, cudaStream_t st) {
  const int grid = fused_grid();
  if (grid <= 0) return cudaErrorNotSupported;
  const int M = p.B;  // S = 1: one row per sequence
  const int QKV = (p.H + 2 * p.G) * p.D;
  if (M <= 0 || p.D != DT_D || p.sync == nullptr || p.d % 8 != 0) return cudaErrorInvalidValue;
  FusedMaps m;
  FusedArgs a;
  RowNorm norm_x;
  norm_x.ss_in = p.ss_x;
  norm_x.eps = p.eps;
  norm_x.d = p.d;
  RowNorm norm_h;
  norm_h.ss_in = p.ss_h;
  norm_h.ss_out = p.ss_h;
  norm_h.eps = p.eps;
  norm_h.d = p.d;
  QkvScatter sc;
  sc.table = p.rope;
  sc.table_seq = p.rope_seq;
  sc.q = p.q;
  sc.kc = p.kc;
  sc.vc = p.vc;
  sc.S = 1;
  sc.start_pos = p.start_pos;
  sc.H = p.H;
  sc.G = p.G;
  sc.D = p.D;
  sc.cache_seq = p.cache_seq;
  sc.halves = p.halves;
  cudaError_t e = gemm_tc_prepare(p.x, p.wqkv, nullptr, nullptr, M, QKV, p.d, EPI_QKV_ROPE, p.status, &p.gemm,
                                  &norm_x, &sc, true, &m.qkv_a, &m.qkv_w, &a.qkv, &a.bn_qkv, false);
  if (e == cudaSuccess)
    e = attn_decode_tc_prepare(p.q, p.kc, p.vc, p.o, p.B, p.start_pos, p.H, p.G, p.cache_seq, p.attn, p.status, &m.q,
                               &m.k, &m.v, &a.attn);
  if (e == cudaSuccess)
    e = gemm_tc_prepare(p.o, p.wo, p.x, p.h, M, p.d, p.H * p.D, EPI_RESIDUAL_SQSUM, p.status, &p.gemm, &norm_h,
                        nullptr, true, &m.o_a, &m.o_w, &a.o, &a.bn_o, false);
  if (e == cudaSuccess)
    e = gemm_tc_prepare(p.h, p.w_gu, nullptr, p.act, M, 2 * p.F, p.d, EPI_SWIGLU_ROWSCALE, p.status, &p.gemm, &norm_h,
                        nullptr, true, &m.gu_a, &m.gu_w, &a.gu, &a.bn_gu, false);
  if (e == cudaSuccess)
    e = gemm_tc_prepare(p.act, p.w_down, p.h, p.y, M, p.d, p.F, EPI_RESIDUAL, p.status, &p.gemm, nullptr, nullptr,
                        true, &m.dn_a, &m.dn_w, &a.dn, &a.bn_dn, false);
  if (e != cudaSuccess) return e;
  a.x = p.x;
  a.ss_x = p.ss_x;
  a.ss_h = p.ss_h;
  a.rows = M;
  a.d = p.d;
  a.sync = p.sync;
  e = cudaMemsetAsync(p.sync, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(FUSED_THREADS);
  cfg.dynamicSmemBytes = FUSED_SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, decode_block_fused_kernel, m, a);
}

}  // namespace llama
