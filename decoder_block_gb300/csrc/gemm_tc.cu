// Persistent, warp-specialised tcgen05 GEMM for the four dense projections of
// the block (QKV, O, gate/up, down) and the LM head:  C = epi(A W^T), with A
// [M,K] activations and W [N,K] nn.Linear weights, both bf16 and K-major.
//
// Per CTA (one per SM, 192 threads), output tiles of 128 x BN (BN = 256, 128
// or 64, picked per shape on the host):
//   warp 0      TMA producer: 128x64 A box + BNx64 W box per stage, 128-byte
//               swizzle, a ring of STAGES shared-memory buffers (deeper for
//               narrower tiles);
//   warp 1      allocates 2*BN TMEM columns, issues tcgen05.mma (M=128, N=BN,
//               K=16) from one thread into one of two BN-column fp32
//               accumulators, commits stage releases and accumulator-ready;
//   warps 2..5  epilogue: tcgen05.ld the accumulator rows of their TMEM lane
//               quarter, apply the fused epilogue (store / + residual /
//               SiLU(gate) * up / fp32 out / RMSNorm row scale / RoPE and
//               KV-cache scatter) and store to global memory, then
//               hand the accumulator back -- overlapping the next tile's K loop.
// Split-K (for few output tiles, e.g. the decode step's M = 64 rows, so that
// every SM streams a share of the weights): a work unit is (tile, K split);
// each epilogue warp adds its 32-row fp32 partial into the tile's fp32
// accumulator in the workspace (vector reductions at L2), counts arrivals on a
// per-(tile, quarter) counter, and the last arriving warp reads the sums back
// once, applies the epilogue and returns the accumulator and the counter to
// zero, so the scratch needs no clearing between launches.
// Launched as a programmatic dependent: for weights the library owns (written
// once at create, by no kernel of a forward) the producer requests the first
// stages' weights before it waits for the previous kernel; everything else
// (activations, residuals, row statistics, outputs) is touched after the wait.
// Every mbarrier wait is bounded (clock budget); on expiry the kernel records a
// status code, drains in-flight copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int NUM_THREADS = 192;
constexpr int GROUP_M = 16;

template <int BN_>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators (128, 256 or 512: powers of two)
};

struct GemmArgs {
  const bf16 *R;
  void *C;
  int M, N, K;
  int *status;
  int splits;        // K splits of each split tile (1: no split)
  int ksteps_split;  // BK steps per split
  int split_tiles;   // the last split_tiles tiles (raster order) are split; their pieces are the first units
  float *part;       // split-K accumulators [tiles][BM][BN] fp32 (zero at launch; left zero at exit)
  int *counters;     // split-K arrivals [tiles][4] (zero at launch; left zero at exit)
  const float *ss_in;  // ROWSCALE epilogues: per-row sum of squares of A's rows
  float *ss_out;       // EPI_RESIDUAL_SQSUM: per-row sum of squares of C (accumulated)
  float inv_d, eps;    // RMSNorm: scale = rsqrt(ss * inv_d + eps)
  QkvScatter qkv;      // EPI_QKV_ROPE destinations
  int prefetch_w;      // W is written by no kernel: load it before the grid dependency wait
  // grouped mode (one GEMM per group, e.g. per expert): rows [group_off[g],
  // group_off[g+1]) of A multiply rows [g * N, (g+1) * N) of W; offsets live on
  // the device (written by an earlier kernel), so the tile count is found there
  const int *group_off;
  int n_groups;
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

// Columns n .. n+15 of row m (EPI_STORE / EPI_RESIDUAL / EPI_F32OUT).  With
// SQSUM, returns the sum of squares of the bf16 values stored.
// Residual of columns n .. n+31 of row m as four 16-byte vectors, loaded ahead of its
// epilogue chunk (vec false: the row is out of range or the columns are not whole; the
// epilogue then loads what it needs itself).
__device__ __forceinline__ void load_residual32(const GemmArgs &a, int m, int n, uint4 (&r)[4], bool &vec) {
  vec = m < a.M && n + 32 <= a.N && (a.N & 7) == 0;
  if (vec) {
    const uint4 *p = reinterpret_cast<const uint4 *>(a.R + (size_t)m * a.N + n);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = p[i];
  }
}

template <int EPI, bool SQSUM = false>
__device__ __forceinline__ float epilogue_chunk16(const float *v, const GemmArgs &a, int m, int n,
                                                  const uint4 *res = nullptr) {
  if (m >= a.M || n >= a.N) return 0.f;
  const size_t base = (size_t)m * a.N + n;
  float sq = 0.f;
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
        uint4 r0 = res != nullptr ? res[0] : *reinterpret_cast<const uint4 *>(r);
        uint4 r1 = res != nullptr ? res[1] : *reinterpret_cast<const uint4 *>(r + 8);
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
    if constexpr (SQSUM) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float q = __bfloat162float(__float2bfloat16_rn(w[i]));
        if (vec || n + i < a.N) sq = fmaf(q, q, sq);
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
  return sq;
}

// Accumulator columns n .. n+31 of row m through the fused epilogue.  For
// SwiGLU the 32 columns are 16 gate then 16 up rows of the interleaved weight.
// Returns the row's sum-of-squares contribution (EPI_RESIDUAL_SQSUM), else 0.
// EPI_QKV_ROPE: 32 consecutive columns of one head (D % 32 == 0), already row
// scaled.  Interleaved pairs (2i, 2i+1) sit in adjacent registers.
__device__ __forceinline__ void qkv_rope_chunk32(const float (&v)[32], const GemmArgs &a, int m, int n) {
  const QkvScatter &r = a.qkv;
  if (m >= a.M || n >= a.N) return;
  const int head = n / r.D, e = n % r.D;
  const int b = m / r.S, p = r.start_pos + m % r.S;
  uint32_t w[16];
  if (head < r.H + r.G) {
    // "The Evolving Transformer 04 · LLaMA", §02 RoPE: (a cos - b sin, a sin + b cos)
    const float4 *cs = reinterpret_cast<const float4 *>(r.table + (size_t)p * (r.D / 2) + e / 2);
    if (r.halves) {
      // pairs (i, i + D/2), i = e/2 .. e/2 + 15: first members to i, second to i + D/2
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 c = __ldg(cs + k);
        const float a0 = v[4 * k], b0 = v[4 * k + 1], a1 = v[4 * k + 2], b1 = v[4 * k + 3];
        lo[k] = pack_bf16(a0 * c.x - b0 * c.y, a1 * c.z - b1 * c.w);
        hi[k] = pack_bf16(a0 * c.y + b0 * c.x, a1 * c.w + b1 * c.z);
      }
      bf16 *base = head < r.H ? r.q + (size_t)m * r.H * r.D + head * r.D
                              : r.kc + (((size_t)b * r.G + (head - r.H)) * r.cache_seq + p) * r.D;
      uint4 *d_lo = reinterpret_cast<uint4 *>(base + e / 2);
      uint4 *d_hi = reinterpret_cast<uint4 *>(base + r.D / 2 + e / 2);
      d_lo[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      d_lo[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      d_hi[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      d_hi[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      return;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 c = __ldg(cs + k);  // {cos_i, sin_i, cos_i+1, sin_i+1}
      const float a0 = v[4 * k], b0 = v[4 * k + 1], a1 = v[4 * k + 2], b1 = v[4 * k + 3];
      w[2 * k] = pack_bf16(a0 * c.x - b0 * c.y, a0 * c.y + b0 * c.x);
      w[2 * k + 1] = pack_bf16(a1 * c.z - b1 * c.w, a1 * c.w + b1 * c.z);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = pack_bf16(v[2 * k], v[2 * k + 1]);
  }
  bf16 *dst;
  if (head < r.H) {
    dst = r.q + (size_t)m * r.H * r.D + n;
  } else {
    const bool is_k = head < r.H + r.G;
    const int g = head - r.H - (is_k ? 0 : r.G);
    dst = (is_k ? r.kc : r.vc) + (((size_t)b * r.G + g) * r.cache_seq + p) * r.D + e;
  }
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d4[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

template <int EPI>
__device__ __forceinline__ float epilogue_chunk32(float (&v)[32], const GemmArgs &a, int m, int n,
                                                  const uint4 *res = nullptr) {
  if constexpr (EPI == EPI_STORE_ROWSCALE || EPI == EPI_SWIGLU_ROWSCALE || EPI == EPI_QKV_ROPE ||
                EPI == EPI_F32OUT_ROWSCALE) {
    // RMSNorm of A's row m, applied to the GEMM result (the gain is folded into W)
    const float r = m < a.M ? rsqrtf(a.ss_in[m] * a.inv_d + a.eps) : 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= r;
  }
  if constexpr (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_ROWSCALE) {
    const int nout = a.N / 2;
    const int f = n / 2;
    if (m < a.M && f < nout) {
      bf16 *dst = reinterpret_cast<bf16 *>(a.C) + (size_t)m * nout + f;
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = pack_bf16(silu_f32(v[2 * i]) * v[16 + 2 * i], silu_f32(v[2 * i + 1]) * v[16 + 2 * i + 1]);
      *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return 0.f;
  } else if constexpr (EPI == EPI_QKV_ROPE) {
    qkv_rope_chunk32(v, a, m, n);
    return 0.f;
  } else if constexpr (EPI == EPI_F32OUT_ROWSCALE) {
    epilogue_chunk16<EPI_F32OUT>(v, a, m, n);
    epilogue_chunk16<EPI_F32OUT>(v + 16, a, m, n + 16);
    return 0.f;
  } else if constexpr (EPI == EPI_STORE_ROWSCALE) {
    epilogue_chunk16<EPI_STORE>(v, a, m, n);
    epilogue_chunk16<EPI_STORE>(v + 16, a, m, n + 16);
    return 0.f;
  } else if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
    return epilogue_chunk16<EPI_RESIDUAL, true>(v, a, m, n, res) +
           epilogue_chunk16<EPI_RESIDUAL, true>(v + 16, a, m, n + 16, res != nullptr ? res + 2 : nullptr);
  } else {
    epilogue_chunk16<EPI>(v, a, m, n, res);
    epilogue_chunk16<EPI>(v + 16, a, m, n + 16, res != nullptr ? res + 2 : nullptr);
    return 0.f;
  }
}

// Tiles of the grouped mode: group g has ceil(rows_g / BM) x n_tiles tiles,
// enumerated group by group, N-tile-major within a group (the m-tiles of one
// weight tile run back to back).
struct GroupedTiles {
  const int *off;
  int n_groups, n_tiles;
  __device__ int count() const {
    int t = 0;
    for (int g = 0; g < n_groups; ++g) t += (off[g + 1] - off[g] + BM - 1) / BM * n_tiles;
    return t;
  }
  __device__ void coords(int u, int &g, int &mt, int &nt) const {
    for (g = 0; g < n_groups; ++g) {
      const int mtg = (off[g + 1] - off[g] + BM - 1) / BM;
      if (u < mtg * n_tiles) {
        nt = u / mtg;
        mt = u % mtg;
        return;
      }
      u -= mtg * n_tiles;
    }
    g = n_groups - 1;
    mt = nt = 0;
  }
};

template <int EPI, int BN, bool GROUPED = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs args) {
  using G = GemmCfg<BN>;
  constexpr int STAGES = G::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * G::STAGE_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + G::NUM_BARS);
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
  const int k_steps = (args.K + BK - 1) / BK;
  const GroupedTiles gt{args.group_off, args.n_groups, n_tiles};
  if constexpr (GROUPED) grid_dependency_wait();  // every role reads the group offsets
  const int num_tiles = m_tiles * n_tiles;
  const int split_units = GROUPED ? 0 : args.split_tiles * args.splits;
  const int num_units = GROUPED ? gt.count() : split_units + (num_tiles - args.split_tiles);
  // unit -> first A row, first W row, end of the valid A rows, N tile, K range in BK steps.
  // Units [0, split_units) are the K pieces of the last split_tiles tiles (spread over
  // every CTA first, so their reductions overlap the whole tiles that follow); the rest
  // are whole tiles.  slot: the split tile's accumulator / counter index, -1 if whole.
  auto unit_coords = [&](int u, int &a_row, int &w_row, int &m_end, int &nt, int &k0, int &k1, int &slot) {
    if constexpr (GROUPED) {
      int g, mt;
      gt.coords(u, g, mt, nt);
      a_row = args.group_off[g] + mt * BM;
      m_end = min(args.group_off[g + 1], args.M);  // never past A, whatever the offsets say
      w_row = g * args.N + nt * BN;
      k0 = 0;
      k1 = k_steps;
      slot = -1;
    } else {
      int tile;
      if (u < split_units) {
        slot = u / args.splits;
        tile = num_tiles - args.split_tiles + slot;
        k0 = (u % args.splits) * args.ksteps_split;
        k1 = min(k_steps, k0 + args.ksteps_split);
      } else {
        slot = -1;
        tile = u - split_units;
        k0 = 0;
        k1 = k_steps;
      }
      int mt;
      tile_coords(tile, m_tiles, n_tiles, mt, nt);
      a_row = mt * BM;
      m_end = args.M;
      w_row = nt * BN;
    }
  };

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
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), G::TMEM_COLS);
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

  allow_dependents_launch();
  if (warp == 0) {
    if (lane == 0) {
      // The weights of the first unit's first stages depend on no earlier
      // kernel: request them before waiting for the activations.
      int pre = 0;
      if (!GROUPED && args.prefetch_w && (int)blockIdx.x < num_units) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(blockIdx.x, a_row, w_row, m_end, nt, k0, k1, slot);
        pre = min(STAGES, k1 - k0);
        for (int i = 0; i < pre; ++i) {
          const uint32_t sb = smem0 + i * G::STAGE_BYTES + G::A_BYTES;
          ptx::mbar_arrive_expect_tx(full_bar(i), G::STAGE_BYTES);
          ptx::tma_load_2d(sb, &tmB, (k0 + i) * BK, w_row, full_bar(i));
        }
      }
      if constexpr (!GROUPED) grid_dependency_wait();
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
        for (int k = k0; k < k1; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const uint32_t sa = smem0 + s * G::STAGE_BYTES, sb = sa + G::A_BYTES;
          if (it < pre) {  // stage s is fresh and its weights are already on the way
            ptx::tma_load_2d(sa, &tmA, k * BK, a_row, full_bar(s));
            ++it;
            continue;
          }
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1, abort_flag, args.status, DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full_bar(s), G::STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmA, k * BK, a_row, full_bar(s));
          ptx::tma_load_2d(sb, &tmB, k * BK, w_row, full_bar(s));
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
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++tcount) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!ptx::mbar_wait(tempty_bar(acc), aph ^ 1, abort_flag, args.status, DEV_TIMEOUT_MMA)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int k = k0; k < k1; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!ptx::mbar_wait(full_bar(s), ph, abort_flag, args.status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = smem0 + s * G::STAGE_BYTES, sb = sa + G::A_BYTES;
          const uint64_t adesc = ptx::smem_desc_sw128(sa), bdesc = ptx::smem_desc_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16_ss(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                             (k > k0 || kk != 0) ? 1u : 0u);
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
    if constexpr (!GROUPED) grid_dependency_wait();  // the epilogue reads R / row statistics and writes C
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int tcount = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++tcount) {
      int a_row, w_row, m_end, nt, k0, k1, slot;
      unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      bool ok = ptx::mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, DEV_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      // rows past the tile's valid range (the next group's rows, or past M) are
      // passed as row M, which every epilogue skips
      const int m = a_row + row < m_end ? a_row + row : args.M;
      if (slot < 0) {
        float sq = 0.f;
        if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_SQSUM) {
          // the next chunk's residual is loaded while this chunk is finished
          uint4 rc[4], rn[4];
          bool vc, vn = false;
          load_residual32(args, m, nt * BN, rc, vc);
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {
            if (c + 32 < BN) load_residual32(args, m, nt * BN + c + 32, rn, vn);
            float v[32];
            ptx::tmem_ld32(trow + c, v);
            sq += epilogue_chunk32<EPI>(v, args, m, nt * BN + c, vc ? rc : nullptr);
#pragma unroll
            for (int i = 0; i < 4; ++i) rc[i] = rn[i];
            vc = vn;
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {
            float v[32];
            ptx::tmem_ld32(trow + c, v);
            sq += epilogue_chunk32<EPI>(v, args, m, nt * BN + c);
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty_bar(acc));
        if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
          if (m < args.M) atomicAdd(args.ss_out + m, sq);
        }
      } else {
        // split-K: add this warp's 32 x BN fp32 partial into the tile's accumulator,
        // release TMEM, count arrivals; the last split's warp finishes the tile
        const int tile = slot;
        const bool rows_live = a_row + q * 32 < args.M;
        float *acc_row = args.part + ((size_t)tile * BM + row) * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          ptx::tmem_ld32(trow + c, v);
          if (m < args.M) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) ptx::red_add_v4(acc_row + c + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(tempty_bar(acc));
        if (rows_live) {
          __threadfence();
          __syncwarp();
          int prev = 0;
          if (lane == 0) prev = atomicAdd(args.counters + tile * 4 + q, 1);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          if (prev == args.splits - 1) {  // every split has added its partial: finish the tile
            __threadfence();
            float sq = 0.f;
            // the next chunk's sums are loaded while this chunk runs its epilogue
            auto load_sums = [&](int c, float (&v)[32]) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 p4 = m < args.M ? __ldcg(reinterpret_cast<const float4 *>(acc_row + c + i))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                v[i] = p4.x;
                v[i + 1] = p4.y;
                v[i + 2] = p4.z;
                v[i + 3] = p4.w;
              }
            };
            // leave the scratch zero for the next launch: this warp is the only
            // reader and every other split has already added its part
            auto clear_sums = [&](int c) {
              if (m < args.M) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                  __stcg(reinterpret_cast<float4 *>(acc_row + c + i), make_float4(0.f, 0.f, 0.f, 0.f));
              }
            };
            constexpr bool kRes = EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_SQSUM;
            float v[32], nx[32];
            uint4 rc[4], rn[4];  // residual of the current / next chunk (residual epilogues)
            bool vc = false, vn = false;
            load_sums(0, v);
            clear_sums(0);
            if (kRes) load_residual32(args, m, nt * BN, rc, vc);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
              if (c + 32 < BN) {
                load_sums(c + 32, nx);
                clear_sums(c + 32);
                if (kRes) load_residual32(args, m, nt * BN + c + 32, rn, vn);
              }
              sq += epilogue_chunk32<EPI>(v, args, m, nt * BN + c, vc ? rc : nullptr);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = nx[i];
#pragma unroll
              for (int i = 0; i < 4; ++i) rc[i] = rn[i];
              vc = vn;
            }
            if (lane == 0) args.counters[tile * 4 + q] = 0;
            if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
              if (m < args.M) atomicAdd(args.ss_out + m, sq);
            }
          }
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, G::TMEM_COLS);
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

template <int EPI, int BN, bool GROUPED = false>
cudaError_t launch_cfg(const bf16 *A, const bf16 *W, GemmArgs args, cudaStream_t st) {
  using G = GemmCfg<BN>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<EPI, BN, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    G::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb;
  const uint64_t w_rows = GROUPED ? (uint64_t)args.N * args.n_groups : (uint64_t)args.N;
  if (!make_map_2d(&ma, A, (uint64_t)args.M, (uint64_t)args.K, BM) ||
      !make_map_2d(&mb, W, w_rows, (uint64_t)args.K, BN))
    return cudaErrorInvalidValue;
  int grid = sm_count();
  if (!GROUPED) {  // grouped: the tile count is on the device; every SM takes part
    const int tiles = ((args.M + BM - 1) / BM) * ((args.N + BN - 1) / BN);
    const int units = args.split_tiles * args.splits + tiles - args.split_tiles;
    grid = units < grid ? units : grid;
  }
  count_launch();
  return launch_pdl(gemm_tc_kernel<EPI, BN, GROUPED>, dim3(grid), dim3(NUM_THREADS), G::SMEM_BYTES, st, ma, mb,
                    args);
}

template <int EPI>
cudaError_t launch_epi(const bf16 *A, const bf16 *W, GemmArgs args, int bn, cudaStream_t st) {
  switch (bn) {
    case 256: return launch_cfg<EPI, 256>(A, W, args, st);
    case 128: return launch_cfg<EPI, 128>(A, W, args, st);
    case 64: return launch_cfg<EPI, 64>(A, W, args, st);
  }
  return cudaErrorInvalidValue;
}

__global__ void permute_halves_rows_kernel(const uint4 *__restrict__ W, uint4 *__restrict__ out, int heads, int D,
                                           int vec_per_row) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t total = (size_t)heads * D * vec_per_row;
  if (idx >= total) return;
  const int orow = (int)(idx / vec_per_row), c = (int)(idx % vec_per_row);
  const int head = orow / D, j = orow % D;
  const int srow = head * D + (j & 1 ? j / 2 + D / 2 : j / 2);
  out[idx] = W[(size_t)srow * vec_per_row + c];
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

cudaError_t launch_gemm_grouped(const bf16 *A, const bf16 *W, void *C, int M, int N, int K, int n_groups,
                                const int *group_off, int epi, int *status, cudaStream_t st) {
  if (M <= 0 || N <= 0 || n_groups <= 0) return cudaSuccess;
  if (K <= 0 || (K & 7) != 0 || group_off == nullptr) return cudaErrorInvalidValue;
  if (epi != EPI_STORE && epi != EPI_SWIGLU) return cudaErrorInvalidValue;
  if (epi == EPI_SWIGLU && (N & 31) != 0) return cudaErrorInvalidValue;
  // a tile never straddles two groups' weights: BN divides N; the widest tile
  // that still gives every SM a tile (counting one tile per 128 rows)
  const int m_tiles = (M + BM - 1) / BM;
  int bn = 0;
  if (N % 256 == 0 && m_tiles * (N / 256) >= sm_count())
    bn = 256;
  else if (N % 128 == 0)
    bn = 128;
  else if (N % 64 == 0)
    bn = 64;
  if (bn == 0) return cudaErrorInvalidValue;
  GemmArgs args{nullptr, C, M, N, K, status, 1, (K + BK - 1) / BK, 0, nullptr, nullptr, nullptr, nullptr, 0.f, 0.f,
                {}, 0, group_off, n_groups};
  if (epi == EPI_STORE) {
    switch (bn) {
      case 256: return launch_cfg<EPI_STORE, 256, true>(A, W, args, st);
      case 128: return launch_cfg<EPI_STORE, 128, true>(A, W, args, st);
      default: return launch_cfg<EPI_STORE, 64, true>(A, W, args, st);
    }
  }
  switch (bn) {
    case 256: return launch_cfg<EPI_SWIGLU, 256, true>(A, W, args, st);
    case 128: return launch_cfg<EPI_SWIGLU, 128, true>(A, W, args, st);
    default: return launch_cfg<EPI_SWIGLU, 64, true>(A, W, args, st);
  }
}

GemmPlan plan_gemm(int M, int N, int K, size_t ws_part_bytes, int ws_counter_slots) {
  const int sms = sm_count();
  const int m_tiles = (M + BM - 1) / BM;
  const int k_steps = (K + BK - 1) / BK;
  GemmPlan p;
  auto tiles_for = [&](int bn) { return m_tiles * ((N + bn - 1) / bn); };
  if (tiles_for(256) >= sms) {
    // Compute-bound regime: fewest waves, weighted by the narrower tiles' lower
    // per-flop efficiency (shared-memory operand traffic per MMA).
    const int bns[3] = {256, 128, 64};
    const double eff[3] = {1.0, 1.12, 1.45};
    double best = 1e30;
    for (int i = 0; i < 3; ++i) {
      const int waves = (tiles_for(bns[i]) + sms - 1) / sms;
      const double cost = waves * bns[i] * eff[i];
      if (cost < best - 1e-9) {
        best = cost;
        p.bn = bns[i];
      }
    }
    // A short partial last wave (at most a quarter of the SMs busy) leaves most SMs
    // idle for a whole tile time: split its tiles along K into pieces that every SM
    // shares (run first, so their reductions overlap the full waves).  The tail then
    // costs ceil(tail * s / sms) / s of a tile time instead of one, plus the pieces'
    // reduction (charged as 0.05 of a tile).  Longer tails gain less than the L2
    // reductions of their many pieces cost (measured), and so do short K loops.
    const int tiles = tiles_for(p.bn), tail = tiles % sms;
    if (tail > 0 && 4 * tail <= sms && k_steps >= 32 && (size_t)tail * BM * p.bn * sizeof(float) <= ws_part_bytes &&
        tail * 4 <= ws_counter_slots) {
      double best_tail = 1.0;
      for (int s = 2; s <= 16 && k_steps / s >= 4; ++s) {
        const double cost = (double)((tail * s + sms - 1) / sms) / s + 0.05;
        if (cost < best_tail - 1e-9) {
          best_tail = cost;
          p.splits = s;
        }
      }
      if (p.splits > 1) {
        p.ksteps_split = (k_steps + p.splits - 1) / p.splits;
        p.splits = (k_steps + p.ksteps_split - 1) / p.ksteps_split;
        p.split_tiles = tail;
      }
    }
    return p;
  }
  // Few output tiles (decode: weight streaming): pick the tile width and K split
  // that minimise the per-SM load, rounds x (K steps per unit) x (shared-memory
  // fill per K step: 16 KB of A plus BN x 128 B of weights); ties go to more
  // units (more SMs streaming weights at once).
  double best = 1e30;
  int best_units = 0;
  const int bns[3] = {256, 128, 64};
  for (int i = 0; i < 3; ++i) {
    const int bn = bns[i];
    const int tiles = tiles_for(bn);
    for (int want = 1; want <= 16 && want <= k_steps; ++want) {
      const int kss = (k_steps + want - 1) / want;
      const int splits = (k_steps + kss - 1) / kss;
      const int units = tiles * splits;
      if (splits > 1 && ((size_t)tiles * BM * bn * sizeof(float) > ws_part_bytes || tiles * 4 > ws_counter_slots))
        continue;
      const int rounds = (units + sms - 1) / sms;
      // + 12 K steps of fixed per-unit cost (pipeline fill, epilogue; measured on the
      // decode shapes); each split piece's reduction into the tile's accumulator
      // (L2 atomics on the same lines, then the last piece's serial finish) adds
      // about two rows of weights' worth per piece (measured on the decode shapes:
      // 9 pieces of a 256-wide tile lose to 4 of a 128-wide one)
      const double cost = (double)rounds * (kss + 12) * (16.0 + bn / 8.0) + (splits > 1 ? splits * bn / 4.0 : 0.0);
      if (cost < best - 1e-9 || (cost <= best + 1e-9 && units > best_units && units <= sms)) {
        best = cost;
        best_units = units;
        p.bn = bn;
        p.splits = splits;
        p.ksteps_split = kss;
      }
    }
  }
  if (p.splits == 1) p.ksteps_split = 0;
  p.split_tiles = p.splits > 1 ? tiles_for(p.bn) : 0;
  return p;
}

size_t gemm_splitk_part_bytes() {
  // Split plans arise only when fewer than one wave of 128x256 tiles exists,
  // i.e. fewer than 2 x SMs 128-wide or 4 x SMs 64-wide tiles: one fp32
  // accumulator tile each.
  return (size_t)sm_count() * BM * 256 * sizeof(float);
}

int gemm_splitk_counter_slots() { return 4 * sm_count() * 4; }

cudaError_t launch_gemm_tc(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                           int *status, cudaStream_t st, const GemmWorkspace *ws, const RowNorm *norm,
                           const QkvScatter *scatter, bool weights_static) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (K <= 0 || (K & 7) != 0) return cudaErrorInvalidValue;
  if ((epi == EPI_SWIGLU || epi == EPI_SWIGLU_ROWSCALE) && (N & 31) != 0) return cudaErrorInvalidValue;
  const bool needs_norm = epi == EPI_STORE_ROWSCALE || epi == EPI_SWIGLU_ROWSCALE || epi == EPI_RESIDUAL_SQSUM ||
                          epi == EPI_QKV_ROPE || epi == EPI_F32OUT_ROWSCALE;
  if (needs_norm && norm == nullptr) return cudaErrorInvalidValue;
  if (epi == EPI_QKV_ROPE) {
    if (scatter == nullptr || scatter->D <= 0 || (scatter->D & 31) != 0 || scatter->S <= 0 ||
        N != (scatter->H + 2 * scatter->G) * scatter->D || M % scatter->S != 0)
      return cudaErrorInvalidValue;
  }
  const GemmPlan plan = plan_gemm(M, N, K, ws != nullptr ? ws->part_bytes : 0, ws != nullptr ? ws->counter_slots : 0);
  GemmArgs args{R, C, M, N, K, status, 1, (K + BK - 1) / BK, 0, nullptr, nullptr, nullptr, nullptr, 0.f, 0.f,
                {}, weights_static ? 1 : 0, nullptr, 0};
  if (scatter != nullptr) args.qkv = *scatter;
  if (norm != nullptr) {
    args.ss_in = norm->ss_in;
    args.ss_out = norm->ss_out;
    args.inv_d = 1.0f / (float)norm->d;
    args.eps = norm->eps;
  }
  if (plan.splits > 1) {
    args.splits = plan.splits;
    args.ksteps_split = plan.ksteps_split;
    args.split_tiles = plan.split_tiles;
    args.part = ws->part;
    args.counters = ws->counters;
  }
  switch (epi) {
    case EPI_STORE: return launch_epi<EPI_STORE>(A, W, args, plan.bn, st);
    case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL>(A, W, args, plan.bn, st);
    case EPI_F32OUT: return launch_epi<EPI_F32OUT>(A, W, args, plan.bn, st);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(A, W, args, plan.bn, st);
    case EPI_STORE_ROWSCALE: return launch_epi<EPI_STORE_ROWSCALE>(A, W, args, plan.bn, st);
    case EPI_SWIGLU_ROWSCALE: return launch_epi<EPI_SWIGLU_ROWSCALE>(A, W, args, plan.bn, st);
    case EPI_RESIDUAL_SQSUM: return launch_epi<EPI_RESIDUAL_SQSUM>(A, W, args, plan.bn, st);
    case EPI_QKV_ROPE: return launch_epi<EPI_QKV_ROPE>(A, W, args, plan.bn, st);
    case EPI_F32OUT_ROWSCALE: return launch_epi<EPI_F32OUT_ROWSCALE>(A, W, args, plan.bn, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_permute_halves_rows(const bf16 *W, bf16 *out, int heads, int D, int d, cudaStream_t st) {
  if ((D & 1) != 0 || (d & 7) != 0) return cudaErrorInvalidValue;
  const int vpr = d / 8;
  const size_t total = (size_t)heads * D * vpr;
  if (total == 0) return cudaSuccess;
  count_launch();
  permute_halves_rows_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const uint4 *>(W), reinterpret_cast<uint4 *>(out), heads, D, vpr);
  return cudaGetLastError();
}

cudaError_t launch_interleave_rows(const bf16 *gate, const bf16 *up, bf16 *out, int F, int d, cudaStream_t st) {
  if ((F & 15) != 0 || (d & 7) != 0) return cudaErrorInvalidValue;
  const int vpr = d / 8;
  const size_t total = (size_t)2 * F * vpr;
  count_launch();
  interleave_rows_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const uint4 *>(gate), reinterpret_cast<const uint4 *>(up), reinterpret_cast<uint4 *>(out), F,
      vpr);
  return cudaGetLastError();
}

}  // namespace llama
