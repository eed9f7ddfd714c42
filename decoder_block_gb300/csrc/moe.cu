// Mixture-of-experts feed-forward: routing, dispatch and combine.
// "Llama 4 From Scratch", MoE (a router sends each token to the top-k of N
// expert feed-forwards; Llama 4 keeps one always-on shared expert); "From
// GPT-2 to Llama: four changes and the reason for each", The feed-forward
// grows a gate (a small layer picks a few feed-forwards per token).
//
// Per forward (T tokens, E experts, top k):
//   router logits  r_t (h W_router^T)          tcgen05 GEMM, fp32 row-scaled epilogue
//   moe_topk       ids / weights per token      this file (one warp per token)
//   moe_offsets    per-expert row offsets       this file (one CTA)
//   moe_dispatch   normalised rows, grouped by expert, into the experts' input
//   expert SwiGLU  grouped tcgen05 GEMMs over the per-expert row ranges
//   moe_combine    y = base + sum_j w_tj * expert output of (t, j)
// The per-expert counters are left zero by moe_offsets for the next forward.
#include <climits>

#include "kernels.h"

namespace llama {
namespace {

__device__ __forceinline__ void argmax_merge(float &v, int &i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

// One warp per token: k rounds of a warp arg-max over the E logits (lowest
// expert id among equal logits; NaN is never picked while another id is
// left), then a softmax over the chosen logits.  counts[e] += 1 per choice.
constexpr int MOE_MAX_E = 256;
__global__ void __launch_bounds__(256) moe_topk_kernel(const float *__restrict__ logits, int ld, int T, int E, int k,
                                                       int *__restrict__ ids, float *__restrict__ wts,
                                                       int *__restrict__ counts) {
  allow_dependents_launch();
  grid_dependency_wait();
  const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  constexpr int PER = MOE_MAX_E / 32;
  float l[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? logits[(size_t)t * ld + e] : -INFINITY;
  }
  unsigned taken = 0;  // bit i: this lane's expert lane + 32 i already chosen
  float first = 0.f, sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken >> i & 1u)) argmax_merge(bv, bi, l[i], e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (bi == INT_MAX) {  // every remaining logit is NaN: take the lowest id not chosen yet
      int lo = INT_MAX;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !(taken >> i & 1u)) lo = min(lo, e);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      bi = lo;
      bv = -INFINITY;
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) first = bv;
    const float p = bv == first ? 1.f : __expf(bv - first);
    sum += p;
    if (lane == 0) {
      ids[(size_t)t * k + j] = bi;
      wts[(size_t)t * k + j] = p;
      atomicAdd(counts + bi, 1);
    }
  }
  __syncwarp();
  if (lane < k) wts[(size_t)t * k + lane] /= sum;
}

// offsets[e] = counts[0] + .. + counts[e-1] (offsets[E] = total); counts and
// fill are left zero.  One CTA of MOE_MAX_E threads.
__global__ void __launch_bounds__(MOE_MAX_E) moe_offsets_kernel(int *__restrict__ counts, int *__restrict__ offsets,
                                                                int *__restrict__ fill, int E) {
  allow_dependents_launch();
  grid_dependency_wait();
  __shared__ int sc[MOE_MAX_E];
  const int e = threadIdx.x;
  const int c = e < E ? counts[e] : 0;
  sc[e] = c;
  __syncthreads();
  // inclusive scan (Hillis-Steele) over MOE_MAX_E entries
  for (int o = 1; o < MOE_MAX_E; o <<= 1) {
    const int add = e >= o ? sc[e - o] : 0;
    __syncthreads();
    sc[e] += add;
    __syncthreads();
  }
  if (e < E) {
    offsets[e + 1] = sc[e];
    counts[e] = 0;
    fill[e] = 0;
  }
  if (e == 0) offsets[0] = 0;
}

// One warp per (token, choice): the slot in its expert's row range, and the
// token's RMSNorm-ed row bf16(h * rsqrt(ss / d + eps) * g) copied there.
__global__ void __launch_bounds__(256) moe_dispatch_kernel(const bf16 *__restrict__ h, const float *__restrict__ ss,
                                                           const bf16 *__restrict__ g, float eps, int T, int d,
                                                           int k, const int *__restrict__ ids,
                                                           const int *__restrict__ offsets, int *__restrict__ fill,
                                                           int *__restrict__ pos, bf16 *__restrict__ xin) {
  allow_dependents_launch();
  grid_dependency_wait();
  const int tj = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (tj >= T * k) return;
  const int t = tj / k;
  int p = 0;
  if (lane == 0) {
    const int e = ids[tj];
    p = offsets[e] + atomicAdd(fill + e, 1);
    if (p < 0 || p >= T * k) p = -1;  // only reachable with corrupted counters: write nothing
    pos[tj] = p < 0 ? 0 : p;
  }
  p = __shfl_sync(0xffffffffu, p, 0);
  if (p < 0) return;
  const float r = rsqrtf(ss[t] / (float)d + eps);
  const bf16 *src = h + (size_t)t * d;
  bf16 *dst = xin + (size_t)p * d;
  for (int c = lane * 8; c < d; c += 32 * 8) {
    Vec16<bf16> x = load16(src + c), gv = load16(g + c), o;
#pragma unroll
    for (int i = 0; i < 8; ++i) o.set(i, x.get(i) * r * gv.get(i));
    store16(dst + c, o);
  }
}

// y[t] = base[t] + sum_j w[t][j] * ye[pos[t][j]] over rows of width d (fp32 sum, bf16 store).
__global__ void __launch_bounds__(256) moe_combine_kernel(const bf16 *__restrict__ base, const bf16 *__restrict__ ye,
                                                          const int *__restrict__ pos, const float *__restrict__ wts,
                                                          int T, int d, int k, bf16 *__restrict__ y) {
  allow_dependents_launch();
  grid_dependency_wait();
  const int nv = d / 8;
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)T * nv) return;
  const int t = (int)(idx / nv), c = (int)(idx % nv) * 8;
  Vec16<bf16> b = load16(base + (size_t)t * d + c);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = b.get(i);
  for (int j = 0; j < k; ++j) {
    const float w = wts[(size_t)t * k + j];
    Vec16<bf16> v = load16(ye + (size_t)pos[(size_t)t * k + j] * d + c);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, v.get(i), acc[i]);
  }
  Vec16<bf16> o;
#pragma unroll
  for (int i = 0; i < 8; ++i) o.set(i, acc[i]);
  store16(y + (size_t)t * d + c, o);
}

}  // namespace

bool moe_supported(int E, int k) { return E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= E && k <= 32; }

cudaError_t launch_moe_topk(const float *logits, int ld, int T, int E, int k, int *ids, float *wts, int *counts,
                            cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (!moe_supported(E, k)) return cudaErrorInvalidValue;
  count_launch();
  return launch_pdl(moe_topk_kernel, dim3((unsigned)(((size_t)T * 32 + 255) / 256)), dim3(256), 0, st, logits, ld, T,
                    E, k, ids, wts, counts);
}

cudaError_t launch_moe_offsets(int *counts, int *offsets, int *fill, int E, cudaStream_t st) {
  if (E < 1 || E > MOE_MAX_E) return cudaErrorInvalidValue;
  count_launch();
  return launch_pdl(moe_offsets_kernel, dim3(1), dim3(MOE_MAX_E), 0, st, counts, offsets, fill, E);
}

cudaError_t launch_moe_dispatch(const bf16 *h, const float *ss, const bf16 *g, float eps, int T, int d, int k,
                                const int *ids, const int *offsets, int *fill, int *pos, bf16 *xin, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (d % 8 != 0) return cudaErrorInvalidValue;
  count_launch();
  return launch_pdl(moe_dispatch_kernel, dim3((unsigned)(((size_t)T * k * 32 + 255) / 256)), dim3(256), 0, st, h, ss,
                    g, eps, T, d, k, ids, offsets, fill, pos, xin);
}

cudaError_t launch_moe_combine(const bf16 *base, const bf16 *ye, const int *pos, const float *wts, int T, int d,
                               int k, bf16 *y, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (d % 8 != 0) return cudaErrorInvalidValue;
  const size_t total = (size_t)T * (d / 8);
  count_launch();
  return launch_pdl(moe_combine_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, st, base, ye, pos, wts,
                    T, d, k, y);
}

}  // namespace llama
