// Launchers of the tcgen05 GEMM (kernel body: gemm_tc_body.cuh): tile-width and
// K-split planning, tensor maps, and the weight re-layouts the epilogues expect.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc_body.cuh"

// 256 x 256 tiles on CTA pairs for large compute-bound GEMMs (tuning define: 0 keeps every GEMM on single CTAs).
#ifndef LLAMA_GEMM_PAIRS
#define LLAMA_GEMM_PAIRS 1
#endif

namespace llama {
namespace {

template <int EPI, int BN, bool GROUPED = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GemmArgs args) {
  gemm_tc_run<EPI, BN, GROUPED>(&tmA, &tmB, args, PhaseSync{});
}

// Whole 256 x 256 tiles on CTA pairs (launched in clusters of two; cta_group::2
// MMAs issued by the even CTA of each pair).
template <int EPI, bool GROUPED = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ GemmArgs args) {
  gemm_tc_run<EPI, 256, GROUPED, true>(&tmA, &tmB, args, PhaseSync{});
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

// Cluster split-K (the K pieces of a tile in one thread-block cluster, summed
// through distributed shared memory) when a plan splits every tile, fits one
// wave of one CTA per SM, and this device can hold all its clusters at once.
// Every CTA of such a grid has exactly one unit.
template <int EPI, int BN>
bool cluster_split_fits(int tiles, int splits, int units) {
  if (splits < 2 || splits > 8 || units != tiles * splits || units > sm_count()) return false;
  static std::mutex mu;
  static int fits[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};  // per cluster size: 0 unknown, then 1 + max clusters
  std::lock_guard<std::mutex> lock(mu);
  if (fits[splits] == 0) {
    // the query needs the kernel's shared-memory opt-in (the kernel may not have run yet)
    cudaFuncSetAttribute(gemm_tc_kernel<EPI, BN, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         GemmCfg<BN>::SMEM_BYTES);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)units);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = GemmCfg<BN>::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<EPI, BN, false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
    fits[splits] = 1 + clusters;
  }
  return fits[splits] - 1 >= tiles;
}

// cluster_split_fits for a tile width chosen at run time (the fit depends on
// the tile width's shared memory, not on the epilogue).
bool cluster_split_fits_bn(int bn, int tiles, int splits, int units) {
  switch (bn) {
    case 256: return cluster_split_fits<EPI_STORE, 256>(tiles, splits, units);
    case 192: return cluster_split_fits<EPI_STORE, 192>(tiles, splits, units);
    case 128: return cluster_split_fits<EPI_STORE, 128>(tiles, splits, units);
    case 64: return cluster_split_fits<EPI_STORE, 64>(tiles, splits, units);
  }
  return false;
}

template <int EPI, int BN, bool GROUPED = false>
cudaError_t launch_cfg(const CUtensorMap &ma, const CUtensorMap &mb, GemmArgs args, cudaStream_t st) {
  using G = GemmCfg<BN>;
  static PerContextOnce smem_limit;
  const cudaError_t attr_err = smem_limit.run([] {
    return cudaFuncSetAttribute(gemm_tc_kernel<EPI, BN, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                G::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int grid = sm_count();
  int cluster = 1;
  if (!GROUPED) {  // grouped: the tile count is on the device; every SM takes part
    const int tiles = ((args.M + BM - 1) / BM) * ((args.N + BN - 1) / BN);
    const int units = args.split_tiles * args.splits + tiles - args.split_tiles;
    grid = units < grid ? units : grid;
    if (args.splits > 1 && args.split_tiles == tiles && cluster_split_fits<EPI, BN>(tiles, args.splits, units)) {
      args.cluster_split = 1;
      cluster = args.splits;
      grid = units;
    }
  }
  count_launch();
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<EPI, BN, GROUPED>, ma, mb, args);
}

// How many clusters of two pair-kernel CTAs the device holds at once (0 when
// the query fails); the pair grid is at most that many pairs, every pair
// resident for the whole launch.  Every pair kernel has the same shared memory
// and thread count, so one of them answers for all.
int pair_slots() {
  static std::mutex mu;
  static int slots = -1;
  static PerContextOnce smem_limit;
  if (smem_limit.run([] {
        return cudaFuncSetAttribute(gemm_tc_pair_kernel<EPI_RESIDUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    GemmCfg<256, true>::SMEM_BYTES);
      }) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (slots < 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = GemmCfg<256, true>::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_pair_kernel<EPI_RESIDUAL>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
    slots = clusters;
  }
  return slots;
}

// GROUPED: the tile count is on the device; every pair takes part.
template <int EPI, bool GROUPED = false>
cudaError_t launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &args, cudaStream_t st) {
  using G = GemmCfg<256, true>;
  static PerContextOnce smem_limit;
  const cudaError_t attr_err = smem_limit.run([] {
    return cudaFuncSetAttribute(gemm_tc_pair_kernel<EPI, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                G::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int pairs = pair_slots();
  if (pairs <= 0) return cudaErrorInvalidConfiguration;
  if (!GROUPED) {
    const int tiles = ((args.M + 2 * BM - 1) / (2 * BM)) * ((args.N + 255) / 256);
    pairs = tiles < pairs ? tiles : pairs;
  }
  count_launch();
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<EPI, GROUPED>, ma, mb, args);
}

template <int EPI>
cudaError_t launch_epi(const CUtensorMap &ma, const CUtensorMap &mb, const GemmArgs &args, int bn, cudaStream_t st) {
  switch (bn) {
    case 256: return launch_cfg<EPI, 256>(ma, mb, args, st);
    case 192: return launch_cfg<EPI, 192>(ma, mb, args, st);
    case 128: return launch_cfg<EPI, 128>(ma, mb, args, st);
    case 64: return launch_cfg<EPI, 64>(ma, mb, args, st);
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
  GemmArgs args{nullptr, C, M, N, K, status, 1, (K + BK - 1) / BK, 0, nullptr, nullptr, nullptr, nullptr, nullptr,
                nullptr, 0.f, 0.f,
                {}, 0, group_off, n_groups};
  CUtensorMap ma, mb;
  // Many rows (at least a wave of 256 x 256 tiles, counted as if in one
  // group) and 256 dividing N: 256-row tiles per group on CTA pairs.
  if (LLAMA_GEMM_PAIRS && N % 256 == 0 && 2 * ((M + 2 * BM - 1) / (2 * BM)) * (N / 256) >= sm_count()) {
    if (!make_map_2d(&ma, A, (uint64_t)M, (uint64_t)K, BM) ||
        !make_map_2d(&mb, W, (uint64_t)N * n_groups, (uint64_t)K, 128))
      return cudaErrorInvalidValue;
    return epi == EPI_STORE ? launch_pair<EPI_STORE, true>(ma, mb, args, st)
                            : launch_pair<EPI_SWIGLU, true>(ma, mb, args, st);
  }
  if (!make_map_2d(&ma, A, (uint64_t)M, (uint64_t)K, BM) ||
      !make_map_2d(&mb, W, (uint64_t)N * n_groups, (uint64_t)K, bn))
    return cudaErrorInvalidValue;
  if (epi == EPI_STORE) {
    switch (bn) {
      case 256: return launch_cfg<EPI_STORE, 256, true>(ma, mb, args, st);
      case 128: return launch_cfg<EPI_STORE, 128, true>(ma, mb, args, st);
      default: return launch_cfg<EPI_STORE, 64, true>(ma, mb, args, st);
    }
  }
  switch (bn) {
    case 256: return launch_cfg<EPI_SWIGLU, 256, true>(ma, mb, args, st);
    case 128: return launch_cfg<EPI_SWIGLU, 128, true>(ma, mb, args, st);
    default: return launch_cfg<EPI_SWIGLU, 64, true>(ma, mb, args, st);
  }
}

GemmPlan plan_gemm(int M, int N, int K, size_t ws_part_bytes, int ws_counter_slots, bool allow_cluster) {
  const int sms = sm_count();
  const int m_tiles = (M + BM - 1) / BM;
  const int k_steps = (K + BK - 1) / BK;
  GemmPlan p;
  auto tiles_for = [&](int bn) { return m_tiles * ((N + bn - 1) / bn); };
  if (tiles_for(256) >= sms) {
    // Compute-bound regime: the fewest waves, counting a split tail (below) as the
    // fraction of a wave it takes, weighted by each tile width's cost per output
    // column.  Every K step brings (128 + BN) x 128 B of operands into an SM, and
    // that delivery, not the MMA, paces a K step (a 128 x 256 step takes about
    // 700 cycles against 512 of MMA); per column it costs 1, 1.11, 1.33 and 2.0
    // times the 256-wide figure for BN = 256, 192, 128, 64.  (Timestamped at the
    // SmolLM2 shape, 64-wide tiles were worse still: 3.4 times per column.)
    const int bns[4] = {256, 192, 128, 64};
    const double eff[4] = {1.0, 1.11, 1.33, 2.0};
    double best = 1e30;
    for (int i = 0; i < 4; ++i) {
      GemmPlan c;
      c.bn = bns[i];
      // A short partial last wave (at most a quarter of the SMs busy) leaves most SMs
      // idle for a whole tile time: split its tiles along K into pieces that every SM
      // shares (run first, so their reductions overlap the full waves).  The tail then
      // costs ceil(tail * s / sms) / s of a tile time instead of one, plus the pieces'
      // reduction (charged as 0.05 of a tile).  Longer tails gain less than the L2
      // reductions of their many pieces cost (measured), and so do short K loops.
      const int tiles = tiles_for(c.bn), tail = tiles % sms;
      double waves = (double)(tiles / sms) + (tail > 0 ? 1.0 : 0.0);
      if (tail > 0 && 4 * tail <= sms && k_steps >= 32 &&
          (size_t)tail * BM * c.bn * sizeof(float) <= ws_part_bytes && tail * 4 <= ws_counter_slots) {
        double best_tail = 1.0;
        for (int sp = 2; sp <= 16 && k_steps / sp >= 4; ++sp) {
          const double tc = (double)((tail * sp + sms - 1) / sms) / sp + 0.05;
          if (tc < best_tail - 1e-9) {
            best_tail = tc;
            c.splits = sp;
          }
        }
        if (c.splits > 1) {
          c.ksteps_split = (k_steps + c.splits - 1) / c.splits;
          c.splits = (k_steps + c.ksteps_split - 1) / c.ksteps_split;
          c.split_tiles = tail;
          waves = (double)(tiles / sms) + best_tail;
        }
      }
      const double cost = waves * c.bn * eff[i];
      if (cost < best - 1e-9) {
        best = cost;
        p = c;
      }
    }
    return p;
  }
  // Few output tiles (decode: weight streaming): pick the tile width and K split
  // that minimise the per-SM load, rounds x (K steps per unit) x (shared-memory
  // fill per K step: 16 KB of A plus BN x 128 B of weights); ties go to more
  // units (more SMs streaming weights at once).  192-wide tiles serve wide
  // unsplit projections (28672 gate/up rows make 150 of them, one per SM, where
  // 256-wide tiles leave 40 SMs without weights to stream) and cluster splits
  // (the 8B QKV projection: 32 tiles in clusters of 4).
  double best = 1e30;
  int best_units = 0;
  const int bns[4] = {256, 192, 128, 64};
  for (int i = 0; i < 4; ++i) {
    const int bn = bns[i];
    const int tiles = tiles_for(bn);
    for (int want = 1; want <= 16 && want <= k_steps; ++want) {
      const int kss = (k_steps + want - 1) / want;
      const int splits = (k_steps + kss - 1) / kss;
      const int units = tiles * splits;
      // the pieces of every tile fit one wave of thread-block clusters: summed
      // through distributed shared memory (see launch_cfg), not L2
      const bool cluster = allow_cluster && splits > 1 && cluster_split_fits_bn(bn, tiles, splits, units);
      if (bn == 192 && splits > 1 && !cluster) continue;
      if (splits > 1 && ((size_t)tiles * BM * bn * sizeof(float) > ws_part_bytes || tiles * 4 > ws_counter_slots))
        continue;
      const int rounds = (units + sms - 1) / sms;
      // + 12 K steps of fixed per-unit cost (pipeline fill, epilogue; measured on the
      // decode shapes).  Reductions, fitted to the 8B decode projections (M = 64):
      // in L2, each piece's atomics on the tile's lines plus the last piece's serial
      // finish cost about two rows of weights per piece and a fixed hand-over (9
      // pieces of a 256-wide tile lose to 4 of a 128-wide one; 3 pieces in L2 lose
      // to a cluster of 4 at 192 wide, 23.2 vs 21.5 us for QKV); in a cluster the
      // cost grows with the square of its size (8 pieces of a 256-wide tile lose to
      // 4 of a 128-wide one, 31.7 vs 30.9 us for the down projection).
      const double red =
          splits > 1 ? (cluster ? splits * splits * bn / 16.0 : splits * bn / 4.0 + 192.0) : 0.0;
      const double cost = (double)rounds * (kss + 12) * (16.0 + bn / 8.0) + red;
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

cudaError_t gemm_tc_prepare(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                            int *status, const GemmWorkspace *ws, const RowNorm *norm, const QkvScatter *scatter,
                            bool weights_static, CUtensorMap *ma, CUtensorMap *mw, GemmArgs *out, int *bn,
                            bool allow_cluster) {
  if (M <= 0 || N <= 0 || K <= 0 || (K & 7) != 0) return cudaErrorInvalidValue;
  if ((epi == EPI_SWIGLU || epi == EPI_SWIGLU_ROWSCALE) && (N & 31) != 0) return cudaErrorInvalidValue;
  const bool needs_norm = epi == EPI_STORE_ROWSCALE || epi == EPI_SWIGLU_ROWSCALE || epi == EPI_RESIDUAL_SQSUM ||
                          epi == EPI_QKV_ROPE || epi == EPI_F32OUT_ROWSCALE;
  if (needs_norm && norm == nullptr) return cudaErrorInvalidValue;
  if (epi == EPI_QKV_ROPE) {
    if (scatter == nullptr || scatter->D <= 0 || (scatter->D & 31) != 0 || scatter->S <= 0 ||
        N != (scatter->H + 2 * scatter->G) * scatter->D || M % scatter->S != 0)
      return cudaErrorInvalidValue;
  }
  const GemmPlan plan = plan_gemm(M, N, K, ws != nullptr ? ws->part_bytes : 0, ws != nullptr ? ws->counter_slots : 0,
                                  allow_cluster);
  GemmArgs args{R, C, M, N, K, status, 1, (K + BK - 1) / BK, 0, nullptr, nullptr, nullptr, nullptr, nullptr,
                nullptr, 0.f, 0.f,
                {}, weights_static ? 1 : 0, nullptr, 0};
  if (scatter != nullptr) args.qkv = *scatter;
  if (norm != nullptr) {
    args.ss_in = norm->ss_in;
    args.ss_out = norm->ss_out;
    args.zero_a = norm->zero_a;
    args.zero_b = norm->zero_b;
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
  if (!make_map_2d(ma, A, (uint64_t)M, (uint64_t)K, BM) || !make_map_2d(mw, W, (uint64_t)N, (uint64_t)K, plan.bn))
    return cudaErrorInvalidValue;
  *out = args;
  *bn = plan.bn;
  return cudaSuccess;
}

cudaError_t launch_gemm_tc(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                           int *status, cudaStream_t st, const GemmWorkspace *ws, const RowNorm *norm,
                           const QkvScatter *scatter, bool weights_static) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  CUtensorMap ma, mb;
  GemmArgs args;
  int bn = 0;
  const cudaError_t e = gemm_tc_prepare(A, W, R, C, M, N, K, epi, status, ws, norm, scatter, weights_static, &ma, &mb,
                                        &args, &bn);
  if (e != cudaSuccess) return e;
  // Compute-bound GEMMs whose plan takes 256-wide tiles run on CTA pairs when
  // there is at least one wave of 256 x 256 tiles: whole tiles, no K splits.
  const bool pair_epi = epi == EPI_QKV_ROPE || epi == EPI_RESIDUAL_SQSUM || epi == EPI_SWIGLU_ROWSCALE ||
                        epi == EPI_RESIDUAL || epi == EPI_F32OUT;
  if (LLAMA_GEMM_PAIRS && pair_epi && bn == 256 &&
      2 * ((M + 2 * BM - 1) / (2 * BM)) * ((N + 255) / 256) >= sm_count()) {
    args.splits = 1;
    args.split_tiles = 0;
    args.ksteps_split = (K + BK - 1) / BK;
    args.part = nullptr;
    args.counters = nullptr;
    if (!make_map_2d(&mb, W, (uint64_t)N, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    switch (epi) {
      case EPI_QKV_ROPE: return launch_pair<EPI_QKV_ROPE>(ma, mb, args, st);
      case EPI_RESIDUAL_SQSUM: return launch_pair<EPI_RESIDUAL_SQSUM>(ma, mb, args, st);
      case EPI_SWIGLU_ROWSCALE: return launch_pair<EPI_SWIGLU_ROWSCALE>(ma, mb, args, st);
      case EPI_RESIDUAL: return launch_pair<EPI_RESIDUAL>(ma, mb, args, st);
      case EPI_F32OUT: return launch_pair<EPI_F32OUT>(ma, mb, args, st);
    }
  }
  switch (epi) {
    case EPI_STORE: return launch_epi<EPI_STORE>(ma, mb, args, bn, st);
    case EPI_RESIDUAL: return launch_epi<EPI_RESIDUAL>(ma, mb, args, bn, st);
    case EPI_F32OUT: return launch_epi<EPI_F32OUT>(ma, mb, args, bn, st);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(ma, mb, args, bn, st);
    case EPI_STORE_ROWSCALE: return launch_epi<EPI_STORE_ROWSCALE>(ma, mb, args, bn, st);
    case EPI_SWIGLU_ROWSCALE: return launch_epi<EPI_SWIGLU_ROWSCALE>(ma, mb, args, bn, st);
    case EPI_RESIDUAL_SQSUM: return launch_epi<EPI_RESIDUAL_SQSUM>(ma, mb, args, bn, st);
    case EPI_QKV_ROPE: return launch_epi<EPI_QKV_ROPE>(ma, mb, args, bn, st);
    case EPI_F32OUT_ROWSCALE: return launch_epi<EPI_F32OUT_ROWSCALE>(ma, mb, args, bn, st);
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
