// tcgen05 GEMM kernel body and its fused epilogues, shared by the GEMM kernels
// (gemm_tc.cu) and the fused decode-step kernel (decode_fused.cu).
//
// Persistent, warp-specialised tcgen05 GEMM for the four dense projections of
// the block (QKV, O, gate/up, down) and the LM head:  C = epi(A W^T), with A
// [M,K] activations and W [N,K] nn.Linear weights, both bf16 and K-major.
//
// Per CTA (one per SM, 192 threads), output tiles of 128 x BN (BN = 256, 192,
// 128 or 64, picked per shape on the host):
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
// Large compute-bound GEMMs run the PAIR variant instead (gemm_tc_run below):
// 256 x 256 tiles on the two CTAs of a cluster with cta_group::2 MMAs.
// Split-K (for few output tiles, e.g. the decode step's M = 64 rows, so that
// every SM streams a share of the weights): a work unit is (tile, K split);
// each epilogue warp adds its 32-row fp32 partial into the tile's fp32
// accumulator in the workspace (vector reductions at L2), counts arrivals on a
// per-(tile, quarter) counter, and the last arriving warp reads the sums back
// once, applies the epilogue and returns the accumulator and the counter to
// zero, so the scratch needs no clearing between launches.
// Launched as a programmatic dependent (or run as a phase of the fused decode
// kernel, phase_sync.cuh): for weights the library owns (written once at
// create, by no kernel of a forward) the producer requests the first stages'
// weights before it waits for the previous kernel (phase); everything else
// (activations, residuals, row statistics, outputs) is touched after the wait.
// Every mbarrier wait is bounded (the handle's wait budget); on expiry the
// kernel records a status code, drains in-flight copies and MMAs (waits bounded
// by the default budget), frees TMEM and returns.
#pragma once

#include <cuda.h>

#include "kernels.h"
#include "phase_sync.cuh"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {

constexpr int BM = 128, BK = 64;
constexpr int NUM_THREADS = 192;
// Rasterisation: tiles are visited GROUP_M M-tiles tall, so that the CTAs
// working at one time share weight tiles in L2.  Measured on the 8B prefill
// block over 200 power-capped steps: 32 tall is 1 % faster than 16; 64 tall
// moves the least DRAM but ran at lower SM clocks and was 5 % slower.
// (Tuning define.)
#ifndef LLAMA_GEMM_GROUP_M
#define LLAMA_GEMM_GROUP_M 32
#endif
constexpr int GROUP_M = LLAMA_GEMM_GROUP_M;
// CTA pairs: 256-row tiles, so the same 4096 rows of A per group are 16 tiles
// tall.  (Tuning define.)
#ifndef LLAMA_GEMM_PAIR_GROUP_M
#define LLAMA_GEMM_PAIR_GROUP_M 16
#endif
constexpr int PAIR_GROUP_M = LLAMA_GEMM_PAIR_GROUP_M;

// PAIR_: the tile is computed by a CTA pair (cta_group::2 MMAs, M = 256): each
// CTA holds 128 rows of A and half of the BN weight rows per stage.
template <int BN_, bool PAIR_ = false>
struct GemmCfg {
  static constexpr int BN = BN_;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_ROWS = PAIR_ ? BN / 2 : BN;  // weight rows this CTA loads per stage
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = PAIR_ ? 6 : (BN == 256 ? 4 : (BN == 192 ? 5 : (BN == 128 ? 6 : 8)));
  static constexpr int NUM_BARS = 2 * STAGES + 8;
  // after the barriers and flags: the four epilogue warps' 2 KB output stages
  static constexpr int STAGE_OUT_OFF = (STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 + 15) / 16 * 16;
  static constexpr int SMEM_BYTES = 1024 + STAGE_OUT_OFF + 4 * 2048;
  // two accumulators of BN columns, in a power-of-two allocation (128, 256 or 512)
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
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
  float *zero_a, *zero_b;  // EPI_RESIDUAL_SQSUM: rows cleared by N tile 0 (null: none)
  float inv_d, eps;    // RMSNorm: scale = rsqrt(ss * inv_d + eps)
  QkvScatter qkv;      // EPI_QKV_ROPE destinations
  int prefetch_w;      // W is written by no kernel: load it before the grid dependency wait
  // grouped mode (one GEMM per group, e.g. per expert): rows [group_off[g],
  // group_off[g+1]) of A multiply rows [g * N, (g+1) * N) of W; offsets live on
  // the device (written by an earlier kernel), so the tile count is found there
  const int *group_off;
  int n_groups;
  // cluster split-K: the grid is one unit per CTA and each cluster (of `splits`
  // CTAs) holds the K pieces of one tile, summed through distributed shared
  // memory instead of L2 (set by the launcher, never in a fused kernel)
  int cluster_split;
};

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int &mt, int &nt,
                                            int group_m = GROUP_M) {
  const int per_group = group_m * n_tiles;
  const int g = tile / per_group;
  const int first = g * group_m;
  const int gm = min(m_tiles - first, group_m);
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
// cs: the chunk's 16 (cos, sin) pairs from load_rope32.
__device__ __forceinline__ void qkv_rope_chunk32(const float (&v)[32], const GemmArgs &a, int m, int n,
                                                 const float4 (&cs)[8]) {
  const QkvScatter &r = a.qkv;
  if (m >= a.M || n >= a.N) return;
  const int head = n / r.D, e = n % r.D;
  const int b = m / r.S, p = r.start_pos + m % r.S;
  uint32_t w[16];
  if (head < r.H + r.G) {
    // "The Evolving Transformer 04 · LLaMA", §02 RoPE: (a cos - b sin, a sin + b cos)
    if (r.halves) {
      // pairs (i, i + D/2), i = e/2 .. e/2 + 15: first members to i, second to i + D/2
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 c = cs[k];
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
      const float4 c = cs[k];  // {cos_i, sin_i, cos_i+1, sin_i+1}
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
constexpr bool epi_row_scaled() {
  return EPI == EPI_STORE_ROWSCALE || EPI == EPI_SWIGLU_ROWSCALE || EPI == EPI_QKV_ROPE || EPI == EPI_F32OUT_ROWSCALE;
}

// RMSNorm of A's row m, applied to the GEMM result by the row-scaled epilogues
// (the gain is folded into W): rsqrt(mean of squares + eps); 1 for the others.
// Loaded once per row, before the accumulator is ready.
template <int EPI>
__device__ __forceinline__ float row_scale(const GemmArgs &a, int m) {
  if constexpr (epi_row_scaled<EPI>()) return m < a.M ? rsqrtf(a.ss_in[m] * a.inv_d + a.eps) : 0.f;
  return 1.f;
}

// The (cos, sin) pairs of QKV columns n .. n+31 at row m's position, loaded ahead
// of their epilogue chunk (EPI_QKV_ROPE only; value heads and dead rows load nothing).
template <int EPI>
__device__ __forceinline__ void load_rope32(const GemmArgs &a, int m, int n, float4 (&cs)[8]) {
  if constexpr (EPI == EPI_QKV_ROPE) {
    const QkvScatter &r = a.qkv;
    if (m < a.M && n < a.N && n / r.D < r.H + r.G) {
      // grouped table: pair group g of position p at float4 g * table_seq + p
      const float4 *p = reinterpret_cast<const float4 *>(r.table) + (size_t)((n % r.D) / 4) * r.table_seq +
                        (r.start_pos + m % r.S);
#pragma unroll
      for (int k = 0; k < 8; ++k) cs[k] = __ldg(p + (size_t)k * r.table_seq);
    }
  }
}

// rs: row_scale of row m; res: the chunk's residual from load_residual32 (or null);
// cs: the chunk's rotation pairs from load_rope32 (EPI_QKV_ROPE).
template <int EPI>
__device__ __forceinline__ float epilogue_chunk32(float (&v)[32], const GemmArgs &a, int m, int n, float rs,
                                                  const uint4 *res, const float4 (&cs)[8]) {
  if constexpr (epi_row_scaled<EPI>()) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= rs;
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
    qkv_rope_chunk32(v, a, m, n, cs);
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

// EPI_RESIDUAL_SQSUM: the epilogue of N tile 0 clears row m of the zero_a /
// zero_b accumulators (one thread per row).
__device__ __forceinline__ void clear_rows(const GemmArgs &a, int m) {
  if (a.zero_a != nullptr) a.zero_a[m] = 0.f;
  if (a.zero_b != nullptr) a.zero_b[m] = 0.f;
}

// Residual epilogues of whole tiles move the residual in and the result out
// through each epilogue warp's 2 KB shared-memory stage (32 rows x 64 bytes):
// lane l reads or writes 16-byte unit l % 4 of row 8j + l / 4, eight rows of 64
// contiguous bytes per instruction, instead of one row per lane (32 rows per
// instruction, which made the load/store units pace the epilogue).  Unit u of
// row r sits at slot (u + r / 2) % 4, so that both access patterns are free of
// bank conflicts.
__device__ __forceinline__ int stage_slot(int r, int u) { return r * 4 + ((u + (r >> 1)) & 3); }

// Residual columns n .. n+31 of rows rbase + 8j + lane / 4 (j = 0..3), unit lane % 4.
__device__ __forceinline__ void coop_load_residual32(const GemmArgs &a, int rbase, int m_end, int n, int lane,
                                                     uint4 (&g)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = rbase + 8 * j + (lane >> 2);
    g[j] = row < m_end ? *reinterpret_cast<const uint4 *>(a.R + (size_t)row * a.N + n + 8 * (lane & 3))
                       : make_uint4(0, 0, 0, 0);
  }
}

// EPI_RESIDUAL / EPI_RESIDUAL_SQSUM over the BN columns from n0 of a whole tile's
// 32 rows from rbase (this warp's TMEM lanes at trow); every 32-column chunk lies
// inside N and N % 8 == 0.  g: chunk 0's residual from coop_load_residual32.
// Returns the sum of squares of this lane's row of stored values.
template <int EPI, int BN>
__device__ __forceinline__ float residual_tile_staged(const GemmArgs &a, uint32_t trow, uint4 *stage, int rbase,
                                                      int m_end, int n0, int lane, uint4 (&g)[4]) {
  float sq = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
#pragma unroll
    for (int j = 0; j < 4; ++j) stage[stage_slot(8 * j + (lane >> 2), lane & 3)] = g[j];
    __syncwarp();
    uint4 rc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) rc[u] = stage[stage_slot(lane, u)];
    if (c + 32 < BN) coop_load_residual32(a, rbase, m_end, n0 + c + 32, lane, g);  // in flight meanwhile
    __syncwarp();
    float v[32];
    ptx::tmem_ld32(trow + c, v);
    uint32_t w[16];
    const bf16 *rb = reinterpret_cast<const bf16 *>(rc);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float x0 = v[i] + __bfloat162float(rb[i]), x1 = v[i + 1] + __bfloat162float(rb[i + 1]);
      w[i / 2] = pack_bf16(x0, x1);
      if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
        const float q0 = __bfloat162float(__float2bfloat16_rn(x0)), q1 = __bfloat162float(__float2bfloat16_rn(x1));
        sq = fmaf(q0, q0, sq);
        sq = fmaf(q1, q1, sq);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) stage[stage_slot(lane, u)] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 8 * j + (lane >> 2);
      const uint4 val = stage[stage_slot(r, lane & 3)];
      if (rbase + r < m_end)
        *reinterpret_cast<uint4 *>(reinterpret_cast<bf16 *>(a.C) + (size_t)(rbase + r) * a.N + n0 + c + 8 * (lane & 3)) =
            val;
    }
    __syncwarp();
  }
  return sq;
}

// Work unit u of a dense (not grouped) GEMM with tile width bn: the K pieces of
// the last split_tiles tiles (raster order) come first, then whole tiles.
// Gives the first A row, first W row, N tile, K range in BK steps and the split
// slot (-1 for a whole tile).
__device__ __forceinline__ void dense_unit(const GemmArgs &args, int bn, int u, int &a_row, int &w_row, int &nt,
                                           int &k0, int &k1, int &slot) {
  const int m_tiles = (args.M + BM - 1) / BM, n_tiles = (args.N + bn - 1) / bn;
  const int k_steps = (args.K + BK - 1) / BK;
  const int num_tiles = m_tiles * n_tiles;
  const int split_units = args.split_tiles * args.splits;
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
  w_row = nt * bn;
}

// Split-K finish of columns [c_begin, c_end) of row r of split tile `tile`
// (N tile nt; output row mm, args.M when the row is dead): read the summed
// partials once, clear them for the next launch (the caller is their only
// reader and every split has added its part), run the epilogue.  The next
// chunk's sums and residual load while this chunk runs.  Returns the row's sum
// of squares for EPI_RESIDUAL_SQSUM.  Called from one place of the epilogue.
template <int EPI, int BN>
__device__ __forceinline__ float splitk_finish(const GemmArgs &args, int tile, int nt, int r, int mm, int c_begin,
                                            int c_end) {
  float *sums = args.part + ((size_t)tile * BM + r) * BN;
  auto load_sums = [&](int c, float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 p4 = mm < args.M ? __ldcg(reinterpret_cast<const float4 *>(sums + c + i))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
      v[i] = p4.x;
      v[i + 1] = p4.y;
      v[i + 2] = p4.z;
      v[i + 3] = p4.w;
    }
  };
  auto clear_sums = [&](int c) {
    if (mm < args.M) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) __stcg(reinterpret_cast<float4 *>(sums + c + i), make_float4(0.f, 0.f, 0.f, 0.f));
    }
  };
  constexpr bool kRes = EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_SQSUM;
  float sq = 0.f;
  float v[32], nx[32];
  uint4 rc[4], rn[4];  // residual of the current / next chunk (residual epilogues)
  float4 cs[8], csn[8];  // rotation pairs of the current / next chunk (EPI_QKV_ROPE)
  bool vc = false, vn = false;
  const float rs = row_scale<EPI>(args, mm);
  load_sums(c_begin, v);
  clear_sums(c_begin);
  if (kRes) load_residual32(args, mm, nt * BN + c_begin, rc, vc);
  load_rope32<EPI>(args, mm, nt * BN + c_begin, cs);
#pragma unroll 1
  for (int c = c_begin; c < c_end; c += 32) {
    if (c + 32 < c_end) {
      load_sums(c + 32, nx);
      clear_sums(c + 32);
      if (kRes) load_residual32(args, mm, nt * BN + c + 32, rn, vn);
      load_rope32<EPI>(args, mm, nt * BN + c + 32, csn);
    }
    sq += epilogue_chunk32<EPI>(v, args, mm, nt * BN + c, rs, vc ? rc : nullptr, cs);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = nx[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) rc[i] = rn[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = csn[i];
    vc = vn;
  }
  return sq;
}

// Tiles of the grouped mode: group g has ceil(rows_g / BM) x n_tiles tiles,
// enumerated group by group, N-tile-major within a group (the m-tiles of one
// weight tile run back to back).
// tile_rows: BM, or 2 * BM for 256-row tiles on CTA pairs.
struct GroupedTiles {
  const int *off;
  int n_groups, n_tiles, tile_rows;
  __device__ int count() const {
    int t = 0;
    for (int g = 0; g < n_groups; ++g) t += (off[g + 1] - off[g] + tile_rows - 1) / tile_rows * n_tiles;
    return t;
  }
  __device__ void coords(int u, int &g, int &mt, int &nt) const {
    for (g = 0; g < n_groups; ++g) {
      const int mtg = (off[g + 1] - off[g] + tile_rows - 1) / tile_rows;
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

// The GEMM of one launch (or one phase of a fused kernel, see phase_sync.cuh):
// every CTA of the grid runs this with its 192 threads.
//
// PAIR: whole 256 x 256 tiles computed by the two CTAs of a cluster (launched
// with cluster size 2, never as a phase of a fused kernel; dense, or grouped
// with 256-row tiles per group).  CTA r loads rows
// r*128 .. r*128+127 of the tile's A rows and of its 256 weight rows into its
// own shared memory; both CTAs' copies complete on the even (leader) CTA's
// full barriers, whose MMA thread issues cta_group::2 MMAs that read both CTAs'
// operands and write 128 accumulator rows into each CTA's tensor memory.  Its
// commits arrive on the stage-empty and accumulator-full barriers of both CTAs;
// each CTA's epilogue drains its own accumulator rows and hands the
// accumulator back to the leader.  A CTA that gives up also raises its peer's
// abort flag.  Per K step each SM now brings in 32 KB of operands instead of
// 48 KB for the same MMA work.
template <int EPI, int BN, bool GROUPED, bool PAIR = false>
__device__ __forceinline__ void gemm_tc_run(const CUtensorMap *tmA, const CUtensorMap *tmB, const GemmArgs &args,
                                            const PhaseSync sync) {
  static_assert(!PAIR || BN == 256, "CTA pairs compute 256 x 256 tiles");
  using G = GemmCfg<BN, PAIR>;
  constexpr int STAGES = G::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * G::STAGE_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + G::NUM_BARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);  // shared split-K finish
  volatile uint32_t *peer_fills = tmem_slot + 3;  // PAIR: fills the peer's producer issued (exchange at exit)

  const uint32_t smem0 = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t fin_bar = bar0 + 8u * (2 * STAGES + 4);
  // shared split-K finish: every epilogue warp's partial is in (4 arrivals), and
  // the arrival count of the tile is known (1 arrival)
  const uint32_t parts_bar = bar0 + 8u * (2 * STAGES + 5);
  const uint32_t count_bar = bar0 + 8u * (2 * STAGES + 6);
  const uint32_t xchg_bar = bar0 + 8u * (2 * STAGES + 7);  // PAIR: the peer's fill count has arrived

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // PAIR: this CTA's rank in the pair; units are distributed over pairs
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int unit_stride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // the leader's copy of one of this CTA's barriers (PAIR), and raising the peer's abort flag
  auto leader = [&](uint32_t bar) { return ptx::mapa_shared(bar, 0); };
  auto abort_peer = [&]() {
    if constexpr (PAIR) ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_u32((const void *)abort_flag), rank ^ 1u), 1u);
  };
  const int m_tiles = PAIR ? (args.M + 2 * BM - 1) / (2 * BM) : (args.M + BM - 1) / BM;
  const int n_tiles = (args.N + BN - 1) / BN;
  const int k_steps = (args.K + BK - 1) / BK;
  const GroupedTiles gt{args.group_off, args.n_groups, n_tiles, PAIR ? 2 * BM : BM};
  if constexpr (GROUPED) grid_dependency_wait();  // every role reads the group offsets
  const int num_tiles = m_tiles * n_tiles;
  const int split_units = (GROUPED || PAIR) ? 0 : args.split_tiles * args.splits;
  const int num_units = GROUPED ? gt.count() : split_units + (num_tiles - args.split_tiles);
  // unit -> first A row, first W row, end of the valid A rows, N tile, K range in BK steps.
  // Units [0, split_units) are the K pieces of the last split_tiles tiles (spread over
  // every CTA first, so their reductions overlap the whole tiles that follow); the rest
  // are whole tiles.  slot: the split tile's accumulator / counter index, -1 if whole.
  auto unit_coords = [&](int u, int &a_row, int &w_row, int &m_end, int &nt, int &k0, int &k1, int &slot) {
    if constexpr (GROUPED) {
      int g, mt;
      gt.coords(u, g, mt, nt);
      a_row = args.group_off[g] + (PAIR ? mt * 2 * BM + (int)rank * BM : mt * BM);
      m_end = min(args.group_off[g + 1], args.M);  // never past A, whatever the offsets say
      w_row = g * args.N + nt * BN + (PAIR ? (int)rank * (BN / 2) : 0);
      k0 = 0;
      k1 = k_steps;
      slot = -1;
    } else if constexpr (PAIR) {
      int mt;
      tile_coords(u, m_tiles, n_tiles, mt, nt, PAIR_GROUP_M);
      a_row = mt * 2 * BM + (int)rank * BM;
      w_row = nt * BN + (int)rank * (BN / 2);
      m_end = args.M;
      k0 = 0;
      k1 = k_steps;
      slot = -1;
    } else {
      dense_unit(args, BN, u, a_row, w_row, nt, k0, k1, slot);
      m_end = args.M;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), PAIR ? 8 : 128);  // PAIR: one arrival per epilogue warp of both CTAs
    }
    ptx::mbar_init(fin_bar, 1);
    ptx::mbar_init(parts_bar, 4);
    ptx::mbar_init(count_bar, 1);
    ptx::mbar_init(xchg_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1 && !sync.fused()) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), G::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), G::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(tmA);
    ptx::tma_prefetch_desc(tmB);
  }
  ptx::tc_fence_before();
  if constexpr (PAIR)
    ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other's
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = sync.fused() ? sync.tmem : *tmem_slot;

  if (!sync.fused()) allow_dependents_launch();
  if (warp == 0) {
    if (lane == 0) {
      // The weights of the first unit's first stages depend on no earlier
      // kernel: request them before waiting for the activations.
      // PAIR: both CTAs' copies complete on the leader's full barriers; the
      // leader alone arrives there, expecting both CTAs' bytes
      auto expect = [&](int s) {
        if constexpr (PAIR) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(s), 2 * G::STAGE_BYTES);
        } else {
          ptx::mbar_arrive_expect_tx(full_bar(s), G::STAGE_BYTES);
        }
      };
      // with a single row of tiles (decode shapes) every weight tile is read
      // once: it goes into L2 as first to evict
      const bool w_once = !PAIR && args.M <= BM;
      auto load = [&](uint32_t dst, const CUtensorMap *map, int x, int y, int s) {
        if constexpr (PAIR)
          ptx::tma_load_2d_pair(dst, map, x, y, leader(full_bar(s)));
        else if (w_once && map == tmB)
          ptx::tma_load_2d_hint(dst, map, x, y, full_bar(s), ptx::policy_evict_first());
        else
          ptx::tma_load_2d(dst, map, x, y, full_bar(s));
      };
      int pre = 0;
      if (!GROUPED && args.prefetch_w && unit0 < num_units) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(unit0, a_row, w_row, m_end, nt, k0, k1, slot);
        pre = min(STAGES, k1 - k0);
        for (int i = 0; i < pre; ++i) {
          const uint32_t sb = smem0 + i * G::STAGE_BYTES + G::A_BYTES;
          expect(i);
          load(sb, tmB, (k0 + i) * BK, w_row, i);
        }
      }
      int it = 0;
      bool ok = true;
      if constexpr (!GROUPED) {
        if (!phase_wait(sync, args.status)) {
          // inputs never became ready: complete the prefetched stages (reading
          // A's rows, in bounds, whatever they hold) so that they can drain
          *abort_flag = 1;
          ok = false;
          if (pre > 0) {
            int a_row, w_row, m_end, nt, k0, k1, slot;
            unit_coords(unit0, a_row, w_row, m_end, nt, k0, k1, slot);
            for (int i = 0; i < pre; ++i) load(smem0 + i * G::STAGE_BYTES, tmA, (k0 + i) * BK, a_row, i);
          }
          it = pre;
        }
      }
      for (int u = unit0; u < num_units && ok; u += unit_stride) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
        for (int k = k0; k < k1; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const uint32_t sa = smem0 + s * G::STAGE_BYTES, sb = sa + G::A_BYTES;
          if (it < pre) {  // stage s is fresh and its weights are already on the way
            load(sa, tmA, k * BK, a_row, s);
            ++it;
            continue;
          }
          if (!ptx::mbar_wait(empty_bar(s), ph ^ 1, abort_flag, args.status, DEV_TIMEOUT_PRODUCER)) {
            abort_peer();
            ok = false;
            break;
          }
          expect(s);
          load(sa, tmA, k * BK, a_row, s);
          load(sb, tmB, k * BK, w_row, s);
          ++it;
        }
      }
      // Every issued copy must have landed before the CTA can exit.
      if constexpr (PAIR) {
        // A fill completes on the leader's barrier only once the leader has
        // arrived for it and both CTAs' bytes have landed.  The producers
        // exchange their fill counts; for fills that only the other one issued
        // (this one gave up earlier) this one supplies its missing part -- the
        // leader its arrival (expecting the peer's bytes only), the peer its
        // bytes' worth of transaction count -- so that every issued copy can
        // complete.  A producer runs at most STAGES fills ahead of the fills
        // the MMAs have consumed, so the leader then waits for the last STAGES
        // fills, and the exit barrier keeps the peer alive until it has.
        ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_u32((const void *)peer_fills), rank ^ 1u), (uint32_t)it);
        ptx::mbar_arrive_cluster(ptx::mapa_shared(xchg_bar, rank ^ 1u));
        int other = it;
        if (ptx::mbar_wait_cluster(xchg_bar, 0, args.status, DEV_TIMEOUT_PRODUCER)) other = (int)*peer_fills;
        for (int j = it; j < other; ++j) {
          if (rank == 0)
            ptx::mbar_arrive_expect_tx(full_bar(j % STAGES), G::STAGE_BYTES);
          else
            ptx::mbar_complete_tx_cluster(leader(full_bar(j % STAGES)), G::STAGE_BYTES);
        }
        if (rank == 0) {
          const int hi = max(it, other);
          for (int j = max(0, hi - STAGES); j < hi; ++j)
            ptx::mbar_drain(full_bar(j % STAGES), (j / STAGES) & 1, args.status, DEV_TIMEOUT_PRODUCER);
        }
      } else {
        for (int j = it - STAGES < 0 ? 0 : it - STAGES; j < it; ++j)
          ptx::mbar_drain(full_bar(j % STAGES), (j / STAGES) & 1, args.status, DEV_TIMEOUT_PRODUCER);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!PAIR || rank == 0)) {  // PAIR: the leader issues the pair's MMAs
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int u = unit0; u < num_units && ok; u += unit_stride, ++tcount) {
        int a_row, w_row, m_end, nt, k0, k1, slot;
        unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1;
        if (!ptx::mbar_wait(tempty_bar(acc), aph ^ 1, abort_flag, args.status, DEV_TIMEOUT_MMA)) {
          abort_peer();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int k = k0; k < k1; ++k) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!ptx::mbar_wait(full_bar(s), ph, abort_flag, args.status, DEV_TIMEOUT_MMA)) {
            abort_peer();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = smem0 + s * G::STAGE_BYTES, sb = sa + G::A_BYTES;
          const uint64_t adesc = ptx::smem_desc_sw128(sa), bdesc = ptx::smem_desc_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if constexpr (PAIR)
              ptx::mma_bf16_ss_pair(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                                    (k > k0 || kk != 0) ? 1u : 0u);
            else
              ptx::mma_bf16_ss(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                               (k > k0 || kk != 0) ? 1u : 0u);
          }
          if constexpr (PAIR)
            ptx::mma_commit_pair(empty_bar(s), 3);  // frees stage s in both CTAs
          else
            ptx::mma_commit(empty_bar(s));
          ++it;
        }
        if (ok) {
          if constexpr (PAIR)
            ptx::mma_commit_pair(tfull_bar(acc), 3);
          else
            ptx::mma_commit(tfull_bar(acc));
        }
      }
      // Wait until every issued MMA has finished before TMEM / smem go away.
      if constexpr (PAIR)
        ptx::mma_commit_pair(fin_bar, 1);
      else
        ptx::mma_commit(fin_bar);
      ptx::mbar_drain(fin_bar, 0, args.status, DEV_TIMEOUT_MMA);
    }
  } else {
    // the epilogue reads R / row statistics and writes C
    bool inputs_ready = true;
    if constexpr (!GROUPED) inputs_ready = phase_wait_warp(sync, args.status);
    if (!inputs_ready) *abort_flag = 1;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint4 *stage_out = reinterpret_cast<uint4 *>(smem + G::STAGE_OUT_OFF + (warp - 2) * 2048);
    int tcount = 0;
    int shared_splits = 0;  // split units finished jointly so far (phase of parts_bar / count_bar)
    // the accumulator's rows are read: hand it back to the MMA thread (PAIR: one
    // arrival per warp on the leader's barrier)
    auto release_acc = [&](int acc) {
      ptx::tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(leader(tempty_bar(acc)));
      } else {
        ptx::mbar_arrive(tempty_bar(acc));
      }
    };
    for (int u = unit0; u < num_units && inputs_ready; u += unit_stride, ++tcount) {
      int a_row, w_row, m_end, nt, k0, k1, slot;
      unit_coords(u, a_row, w_row, m_end, nt, k0, k1, slot);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1;
      // rows past the tile's valid range (the next group's rows, or past M) are
      // passed as row M, which every epilogue skips
      const int m = a_row + row < m_end ? a_row + row : args.M;
      // A whole tile's row scale and its first chunk's residual and rotation pairs
      // are loaded while its MMAs run: with a short K loop the epilogue is the
      // critical path, and each of these loads would otherwise stall a chunk.
      constexpr bool kRes = EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_SQSUM;
      // whole 32-column chunks of a residual epilogue go through the output stage
      const bool staged = kRes && (args.N & 7) == 0 && (nt + 1) * BN <= args.N;
      float rs = 1.f;
      uint4 rc[4];
      float4 cs[8];
      bool vc = false;
      if (slot < 0) {
        rs = row_scale<EPI>(args, m);
        if (staged)
          coop_load_residual32(args, a_row + q * 32, m_end, nt * BN, lane, rc);
        else if (kRes)
          load_residual32(args, m, nt * BN, rc, vc);
        load_rope32<EPI>(args, m, nt * BN, cs);
      }
      bool ok = ptx::mbar_wait(tfull_bar(acc), aph, abort_flag, args.status, DEV_TIMEOUT_EPILOGUE);
      if (!__all_sync(0xffffffffu, ok)) {
        abort_peer();
        break;
      }
      ptx::tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (slot < 0 && staged) {
        const float sq = residual_tile_staged<EPI, BN>(args, trow, stage_out, a_row + q * 32, m_end, nt * BN, lane, rc);
        release_acc(acc);
        if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
          if (m < args.M) {
            atomicAdd(args.ss_out + m, sq);
            if (nt == 0) clear_rows(args, m);
          }
        }
      } else if (slot < 0) {
        // the next chunk's residual and rotation pairs load while this chunk is finished
        float sq = 0.f;
        uint4 rn[4];
        float4 csn[8];
        bool vn = false;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          if (c + 32 < BN) {
            if (kRes) load_residual32(args, m, nt * BN + c + 32, rn, vn);
            load_rope32<EPI>(args, m, nt * BN + c + 32, csn);
          }
          float v[32];
          ptx::tmem_ld32(trow + c, v);
          sq += epilogue_chunk32<EPI>(v, args, m, nt * BN + c, rs, vc ? rc : nullptr, cs);
          if (kRes) {
#pragma unroll
            for (int i = 0; i < 4; ++i) rc[i] = rn[i];
            vc = vn;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) cs[i] = csn[i];
        }
        release_acc(acc);
        if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
          if (m < args.M) {
            atomicAdd(args.ss_out + m, sq);
            if (nt == 0) clear_rows(args, m);
          }
        }
      } else {
        if (args.cluster_split) {
          // cluster split-K: this CTA's only unit; its fp32 partial goes into the
          // (now idle) stage buffers, [BN / 4][128 rows][4 columns], and the
          // cluster sums the pieces at the end of the kernel
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {
            float v[32];
            ptx::tmem_ld32(trow + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::st_shared_v4(smem0 + (uint32_t)((((c >> 2) + i) * BM + row) * 16), v[4 * i], v[4 * i + 1],
                                v[4 * i + 2], v[4 * i + 3]);
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(tempty_bar(acc));
          continue;
        }
        // split-K: add this warp's 32 x BN fp32 partial into the tile's accumulator,
        // release TMEM, count arrivals; the last split to arrive finishes the tile
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
        // who finishes what: row fin_r of the tile (output row fin_m), columns
        // [fin_c0, fin_c1); cnt_slot: the counter this lane returns to zero
        bool do_fin = false;
        int fin_r = 0, fin_m = args.M, fin_c0 = 0, fin_c1 = 0, cnt_slot = -1;
        if (m_end - a_row > 64) {
          // a full tile: each warp counts its own 32 rows and the last split's warp
          // finishes them
          if (rows_live) {
            ptx::fence_acq_rel_gpu();
            __syncwarp();
            int prev = 0;
            if (lane == 0) prev = atomicAdd(args.counters + tile * 4 + q, 1);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            if (prev == args.splits - 1) {  // every split has added its partial
              do_fin = true;
              fin_r = row;
              fin_m = m;
              fin_c1 = BN;
              cnt_slot = lane == 0 ? tile * 4 + q : -1;
            }
          }
        } else {
          // at most 64 live rows (the decode shapes): the tile's arrivals are
          // counted once per CTA, and the last CTA's four epilogue warps share the
          // finish, 16 rows x half the columns each, instead of one or two warps
          // finishing whole 32-row slices
          ptx::fence_acq_rel_gpu();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(parts_bar);
          const uint32_t sph = shared_splits & 1;
          if (warp == 2) {
            const bool in = ptx::mbar_wait(parts_bar, sph, abort_flag, args.status, DEV_TIMEOUT_EPILOGUE);
            if (lane == 0) {
              const int prev = in ? atomicAdd(args.counters + tile * 4, 1) : -1;
              *last_flag = prev == args.splits - 1 ? 1 : 0;
              ptx::mbar_arrive(count_bar);
            }
            __syncwarp();
          }
          const bool known = ptx::mbar_wait(count_bar, sph, abort_flag, args.status, DEV_TIMEOUT_EPILOGUE);
          ++shared_splits;
          if (__all_sync(0xffffffffu, known) && *last_flag != 0) {
            do_fin = true;
            fin_r = (warp - 2) * 16 + (lane & 15);
            fin_m = a_row + fin_r < m_end ? a_row + fin_r : args.M;
            fin_c0 = (lane >> 4) * (BN / 2);
            fin_c1 = fin_c0 + BN / 2;
            cnt_slot = warp == 2 && lane == 0 ? tile * 4 : -1;
          }
        }
        if (do_fin) {
          ptx::fence_acq_rel_gpu();
          const float sq = splitk_finish<EPI, BN>(args, tile, nt, fin_r, fin_m, fin_c0, fin_c1);
          if (cnt_slot >= 0) args.counters[cnt_slot] = 0;
          if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
            if (fin_m < args.M) {
              atomicAdd(args.ss_out + fin_m, sq);
              if (nt == 0 && fin_c0 == 0) clear_rows(args, fin_m);
            }
          }
        }
      }
    }
  }
  if (!GROUPED && !PAIR && args.cluster_split) {
    // Every CTA of the cluster holds one K piece of the same tile.  Once all
    // partials are in shared memory, CTA `rank` finishes the 32-column chunks
    // rank, rank + splits, ...: each epilogue thread (one tile row) sums the
    // pieces in piece order (the result does not depend on timing) and runs the
    // epilogue.  The second barrier keeps every CTA's shared memory alive until
    // the others have read it.  Both barriers are reached by every thread.
    ptx::cluster_sync();
    if (warp >= 2) {
      int a_row, w_row, nt, k0, k1, slot;
      dense_unit(args, BN, blockIdx.x, a_row, w_row, nt, k0, k1, slot);
      const int r = threadIdx.x - 64;  // tile row
      const int m = a_row + r < args.M ? a_row + r : args.M;
      const uint32_t rank = ptx::cluster_ctarank();
      float sq = 0.f;
      const float rs = row_scale<EPI>(args, m);
      for (int ch = (int)rank; ch < BN / 32 && m < args.M; ch += args.splits) {
        // the chunk's rotation pairs and residual are requested ahead of the piece loads
        float4 cs[8];
        load_rope32<EPI>(args, m, nt * BN + ch * 32, cs);
        uint4 rc[4];
        bool vc = false;
        if constexpr (EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_SQSUM) load_residual32(args, m, nt * BN + ch * 32, rc, vc);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        // the pieces' loads are in flight together (one distributed shared-memory
        // round trip per group of four pieces, not per load), then added in piece order
        for (int p0 = 0; p0 < args.splits; p0 += 4) {
          const int np = min(4, args.splits - p0);
          float4 p4[4][8];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q < np) {
              const uint32_t base = ptx::mapa_shared(smem0, (uint32_t)(p0 + q));
#pragma unroll
              for (int i = 0; i < 8; ++i)
                p4[q][i] = ptx::ld_cluster_v4(base + (uint32_t)((((ch * 32) >> 2) + i) * BM + r) * 16);
            }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q < np) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[4 * i] += p4[q][i].x;
                v[4 * i + 1] += p4[q][i].y;
                v[4 * i + 2] += p4[q][i].z;
                v[4 * i + 3] += p4[q][i].w;
              }
            }
        }
        sq += epilogue_chunk32<EPI>(v, args, m, nt * BN + ch * 32, rs, vc ? rc : nullptr, cs);
      }
      if constexpr (EPI == EPI_RESIDUAL_SQSUM) {
        if (m < args.M) {
          atomicAdd(args.ss_out + m, sq);
          if (nt == 0 && rank == 0) clear_rows(args, m);
        }
      }
    }
    ptx::cluster_sync();
  }
  ptx::tc_fence_before();
  if constexpr (PAIR)
    ptx::cluster_sync();  // neither CTA leaves while the pair's MMAs or copies may still use its memory
  else
    __syncthreads();
  if (sync.fused()) {  // the next phase reuses this shared memory and TMEM
    if (threadIdx.x == 0) {
      for (int i = 0; i < G::NUM_BARS; ++i) ptx::mbar_inval(bar0 + 8u * i);
    }
  } else if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem_base, G::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem_base, G::TMEM_COLS);
  }
}

// Validation, tile plan (plan_gemm), arguments and tensor maps of one GEMM,
// exactly as launch_gemm_tc launches it (arguments as there); bn receives the
// plan's tile width.  For a caller that runs the GEMM as a phase of its own
// kernel (allow_cluster false: a phase cannot use thread-block clusters).  M, N > 0.
cudaError_t gemm_tc_prepare(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                            int *status, const GemmWorkspace *ws, const RowNorm *norm, const QkvScatter *scatter,
                            bool weights_static, CUtensorMap *ma, CUtensorMap *mw, GemmArgs *args, int *bn,
                            bool allow_cluster = true);

}  // namespace llama
