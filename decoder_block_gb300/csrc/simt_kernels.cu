// Portable CUDA-core kernels of the decoder block: RMSNorm, RoPE + KV-cache
// write, embedding gather, and the fp32-accumulating GEMM / attention used by
// the fp32 path (tiny configuration) and as the fallback for shapes the tensor
// core kernels do not cover.
#include "kernels.h"

namespace llama {

// ---------------------------------------------------------------- RMSNorm ---
// "The Evolving Transformer 04 · LLaMA", §03 RMSNorm: x * rsqrt(mean(x^2) + eps) * g.
// One warp per row, 16-byte vectors, fp32 sum of squares.  Rows of up to
// NV * 32 vectors are held in registers (one read of x, one write of out, all
// of a lane's loads in flight together); longer rows take the two-pass loop.
template <typename T, int NV>
__global__ void __launch_bounds__(256) rmsnorm_reg_kernel(const T *__restrict__ x, const T *__restrict__ g,
                                                          T *__restrict__ out, int rows, int d, float eps) {
  constexpr int V = Vec16<T>::N;
  const int row = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T *xr = x + (size_t)row * d;
  T *orow = out + (size_t)row * d;
  const int nv = d / V;
  Vec16<T> v[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int i = lane + 32 * j;
    if (i < nv) v[j] = load16(xr + (size_t)i * V);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (lane + 32 * j < nv) {
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const float f = v[j].get(k);
        ss = fmaf(f, f, ss);
      }
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)d + eps);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int i = lane + 32 * j;
    if (i < nv) {
      const Vec16<T> gv = load16(g + (size_t)i * V);
      Vec16<T> o;
#pragma unroll
      for (int k = 0; k < V; ++k) o.set(k, v[j].get(k) * r * gv.get(k));
      store16(orow + (size_t)i * V, o);
    }
  }
}

template <typename T>
__global__ void rmsnorm_kernel(const T *__restrict__ x, const T *__restrict__ g, T *__restrict__ out, int rows,
                               int d, float eps) {
  constexpr int V = Vec16<T>::N;
  const int row = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T *xr = x + (size_t)row * d;
  T *orow = out + (size_t)row * d;
  const int nv = d / V;
  float ss = 0.f;
#pragma unroll 8
  for (int i = lane; i < nv; i += 32) {
    Vec16<T> v = load16(xr + (size_t)i * V);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      float f = v.get(k);
      ss = fmaf(f, f, ss);
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)d + eps);
#pragma unroll 8
  for (int i = lane; i < nv; i += 32) {
    Vec16<T> v = load16(xr + (size_t)i * V);
    Vec16<T> gv = load16(g + (size_t)i * V);
    Vec16<T> o;
#pragma unroll
    for (int k = 0; k < V; ++k) o.set(k, v.get(k) * r * gv.get(k));
    store16(orow + (size_t)i * V, o);
  }
}

// Long rows: one CTA per row, each thread holding PT of its 16-byte vectors
// (consecutive threads, consecutive vectors) in registers between the sum of
// squares and the scaled store, so the row is read from memory once; the
// warps' partial sums meet in shared memory.  Small CTAs keep many rows in
// flight per SM.
template <typename T, int PT>
__global__ void __launch_bounds__(256) rmsnorm_row_cta_kernel(const T *__restrict__ x, const T *__restrict__ g,
                                                              T *__restrict__ out, int d, float eps) {
  constexpr int V = Vec16<T>::N;
  __shared__ float part[8];
  const T *xr = x + (size_t)blockIdx.x * d;
  T *orow = out + (size_t)blockIdx.x * d;
  const int nv = d / V;
  Vec16<T> v[PT];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < PT; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      v[j] = load16(xr + (size_t)i * V);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const float f = v[j].get(k);
        ss = fmaf(f, f, ss);
      }
    }
  }
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) part[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nwarps; ++w) tot += part[w];
  // "The Evolving Transformer 04 · LLaMA", §03 RMSNorm: x * rsqrt(mean(x^2) + eps) * g
  const float r = rsqrtf(tot / (float)d + eps);
#pragma unroll
  for (int j = 0; j < PT; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nv) {
      const Vec16<T> gv = load16(g + (size_t)i * V);
      Vec16<T> o;
#pragma unroll
      for (int k = 0; k < V; ++k) o.set(k, v[j].get(k) * r * gv.get(k));
      store16(orow + (size_t)i * V, o);
    }
  }
}

template <typename T>
cudaError_t launch_rmsnorm(const T *x, const T *g, T *out, int rows, int d, float eps, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (int)(((size_t)rows * 32 + threads - 1) / threads);
  const int nv = d / Vec16<T>::N;
  const int per_lane = (nv + 31) / 32;
  count_launch();
  // Short rows (up to four 16-byte vectors per lane) stay in one warp's
  // registers between the two halves of the computation.  Longer rows take a
  // CTA each (rmsnorm_row_cta_kernel), again read once.  A warp holding a
  // 4096-wide row in registers needed ~150 registers and one 256-thread CTA
  // per SM, too few loads in flight (32 us at 8192 x 4096 bf16), and reading
  // the row twice, the second time from L2, took 26.6 us.  Rows beyond 2048
  // vectors are read twice (rmsnorm_kernel).
  if (per_lane > 4 && nv <= 8 * 256) {
    // one CTA per row: 128 threads up to 512 vectors, else 256 (at most 8 vectors each)
    const int cta = nv <= 512 ? 128 : 256;
    const int pt = (nv + cta - 1) / cta;
    switch (pt) {
      case 1: rmsnorm_row_cta_kernel<T, 1><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 2: rmsnorm_row_cta_kernel<T, 2><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 3: rmsnorm_row_cta_kernel<T, 3><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 4: rmsnorm_row_cta_kernel<T, 4><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 5: rmsnorm_row_cta_kernel<T, 5><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 6: rmsnorm_row_cta_kernel<T, 6><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      case 7: rmsnorm_row_cta_kernel<T, 7><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
      default: rmsnorm_row_cta_kernel<T, 8><<<rows, cta, 0, st>>>(x, g, out, d, eps); break;
    }
    return cudaGetLastError();
  }
  switch (per_lane) {
    case 1: rmsnorm_reg_kernel<T, 1><<<blocks, threads, 0, st>>>(x, g, out, rows, d, eps); break;
    case 2: rmsnorm_reg_kernel<T, 2><<<blocks, threads, 0, st>>>(x, g, out, rows, d, eps); break;
    case 3: rmsnorm_reg_kernel<T, 3><<<blocks, threads, 0, st>>>(x, g, out, rows, d, eps); break;
    case 4: rmsnorm_reg_kernel<T, 4><<<blocks, threads, 0, st>>>(x, g, out, rows, d, eps); break;
    default: rmsnorm_kernel<T><<<blocks, threads, 0, st>>>(x, g, out, rows, d, eps); break;
  }
  return cudaGetLastError();
}

// Sum of squares per row (the RMSNorm statistic of rows the next GEMM normalises
// in its epilogue): one warp per row, 16-byte loads, fp32 accumulation.  Also
// clears zero_out[row] and zero_out2[row] (accumulators later epilogues add
// into; either may be null), which keeps memsets out of the kernel chain.
__global__ void __launch_bounds__(256) row_sqsum_kernel(const bf16 *__restrict__ x, float *__restrict__ ss,
                                                        float *__restrict__ zero_out, float *__restrict__ zero_out2,
                                                        int rows, int d) {
  allow_dependents_launch();
  grid_dependency_wait();
  const int row = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const bf16 *xr = x + (size_t)row * d;
  const int nv = d / 8;
  float acc = 0.f;
#pragma unroll 4
  for (int i = lane; i < nv; i += 32) {
    Vec16<bf16> v = load16(xr + (size_t)i * 8);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float f = v.get(k);
      acc = fmaf(f, f, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    ss[row] = acc;
    if (zero_out != nullptr) zero_out[row] = 0.f;
    if (zero_out2 != nullptr) zero_out2[row] = 0.f;
  }
}

cudaError_t launch_row_sqsum(const bf16 *x, float *ss, float *zero_out, int rows, int d, cudaStream_t st,
                             float *zero_out2) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  return launch_pdl(row_sqsum_kernel, dim3((unsigned)(((size_t)rows * 32 + 255) / 256)), dim3(256), 0, st, x, ss,
                    zero_out, zero_out2, rows, d);
}

__global__ void scale_columns_kernel(bf16 *__restrict__ W, const bf16 *__restrict__ g, int rows, int cols) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)rows * cols) return;
  const int k = (int)(idx % cols);
  W[idx] = __float2bfloat16_rn(__bfloat162float(W[idx]) * __bfloat162float(g[k]));
}

cudaError_t launch_scale_columns(bf16 *W, const bf16 *g, int rows, int cols, cudaStream_t st) {
  const size_t n = (size_t)rows * cols;
  if (n == 0) return cudaSuccess;
  count_launch();
  scale_columns_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(W, g, rows, cols);
  return cudaGetLastError();
}

// ------------------------------------------------------------ SIMT GEMM ---
// C[M,N] = A[M,K] W[N,K]^T (nn.Linear, no bias), fp32 accumulation.
// 64x64 output tile per 256-thread CTA, 4x4 per thread, K step 16.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <typename T, int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T *__restrict__ A, const T *__restrict__ W,
                                                        const T *__restrict__ W3, const T *__restrict__ R,
                                                        void *__restrict__ C, int M, int N, int K) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Ws[SG_BK][SG_BN + 4];
  __shared__ float W3s[EPI == EPI_SWIGLU ? SG_BK : 1][EPI == EPI_SWIGLU ? SG_BN + 4 : 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  float acc[4][4], acc3[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc3[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += SG_BK) {
    for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
      const int r = i / SG_BK, kk = i % SG_BK;
      const int k = k0 + kk;
      const int m = m0 + r, n = n0 + r;
      As[kk][r] = (m < M && k < K) ? to_f32<T>(A[(size_t)m * K + k]) : 0.f;
      Ws[kk][r] = (n < N && k < K) ? to_f32<T>(W[(size_t)n * K + k]) : 0.f;
      if constexpr (EPI == EPI_SWIGLU) W3s[kk][r] = (n < N && k < K) ? to_f32<T>(W3[(size_t)n * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = W3s[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc3[i][j] = fmaf(a[i], b[j], acc3[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      const size_t idx = (size_t)m * N + n;
      float v = acc[i][j];
      if constexpr (EPI == EPI_RESIDUAL) v += to_f32<T>(R[idx]);
      if constexpr (EPI == EPI_SWIGLU) v = silu_f32(v) * acc3[i][j];
      if constexpr (EPI == EPI_F32OUT)
        reinterpret_cast<float *>(C)[idx] = v;
      else
        reinterpret_cast<T *>(C)[idx] = from_f32<T>(v);
    }
  }
}

template <typename T>
cudaError_t launch_gemm_simt(const T *A, const T *W, const T *W3, const T *R, void *C, int M, int N, int K,
                             int epi, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + SG_BN - 1) / SG_BN, (M + SG_BM - 1) / SG_BM);
  count_launch();
  switch (epi) {
    case EPI_STORE: gemm_simt_kernel<T, EPI_STORE><<<grid, 256, 0, st>>>(A, W, W3, R, C, M, N, K); break;
    case EPI_RESIDUAL: gemm_simt_kernel<T, EPI_RESIDUAL><<<grid, 256, 0, st>>>(A, W, W3, R, C, M, N, K); break;
    case EPI_F32OUT: gemm_simt_kernel<T, EPI_F32OUT><<<grid, 256, 0, st>>>(A, W, W3, R, C, M, N, K); break;
    case EPI_SWIGLU: gemm_simt_kernel<T, EPI_SWIGLU><<<grid, 256, 0, st>>>(A, W, W3, R, C, M, N, K); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ RoPE table ---
// "Mini Llama 2 Implementation", Rotary positional embeddings: angle of pair i
// at position p is p * theta^(-2i/D).  With a scaling factor > 1 the frequency
// is stretched as "From GPT-2 to Llama: four changes and the reason for each",
// Positions become a rotation describes for Llama 3.1: long wavelengths slowed
// by the factor, short ones kept, linear blend in between.  Built once per
// block in fp64, stored fp32.
__device__ double rope_frequency(int i, int D, double theta, RopeScaling sc) {
  const double f = pow(theta, -2.0 * (double)i / (double)D);
  if (!(sc.factor > 1.0)) return f;
  const double lam = 2.0 * 3.14159265358979323846 / f;
  if (lam < sc.original_max_pos / sc.high) return f;
  if (lam > sc.original_max_pos / sc.low) return f / sc.factor;
  const double w = (sc.original_max_pos / lam - sc.low) / (sc.high - sc.low);
  return (1.0 - w) * f / sc.factor + w * f;
}

// grouped: pair i of position p at float2 index ((i / 2) * max_seq + p) * 2 + i % 2
// (launch_rope_table_grouped), else at p * (D / 2) + i.
template <bool GROUPED>
__global__ void rope_table_kernel(float2 *table, int max_seq, int D, double theta, RopeScaling sc) {
  const int half = D / 2;
  const size_t n = (size_t)max_seq * half;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx / half), i = (int)(idx % half);
    const double f = rope_frequency(i, D, theta, sc);
    double s, c;
    sincos((double)p * f, &s, &c);
    const size_t at = GROUPED ? ((size_t)(i / 2) * max_seq + p) * 2 + (i & 1) : idx;
    table[at] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2 *table, int max_seq, int D, double theta, const RopeScaling &sc,
                              cudaStream_t st) {
  const size_t n = (size_t)max_seq * (D / 2);
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  count_launch();
  rope_table_kernel<false><<<blocks > 0 ? blocks : 1, 256, 0, st>>>(table, max_seq, D, theta, sc);
  return cudaGetLastError();
}

cudaError_t launch_rope_table_grouped(float2 *table, int max_seq, int D, double theta, const RopeScaling &sc,
                                      cudaStream_t st) {
  if (D % 4 != 0) return cudaErrorInvalidValue;
  const size_t n = (size_t)max_seq * (D / 2);
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  count_launch();
  rope_table_kernel<true><<<blocks > 0 ? blocks : 1, 256, 0, st>>>(table, max_seq, D, theta, sc);
  return cudaGetLastError();
}

// ------------------------------------------------------ RoPE + KV write ---
// Each thread owns one 16-byte vector of a token's fused [q | k | v] row; a
// vector never straddles a head (D % 8 == 0).  Interleaved layout: the vector
// holds whole (2i, 2i+1) pairs.  Halves layout: the thread of a vector in the
// first half of a q / k head also loads the matching vector D/2 further on and
// writes both (pairs (i, i + D/2)); threads of second-half vectors have nothing
// to do.  q: rotated into q_out; k: rotated into the K cache at position
// start_pos + s; v: copied into the V cache ("Full Llama 3 transformer block",
// How it works: RoPE rotates Q and K, keys/values are written into a cache).
template <typename T>
__global__ void __launch_bounds__(256) rope_kv_kernel(const T *__restrict__ qkv, T *__restrict__ q_out,
                                                      T *__restrict__ kc, T *__restrict__ vc,
                                                      const float2 *__restrict__ table, int t0, int S,
                                                      int start_pos, int H, int G, int D, int cache_seq, int halves) {
  // grid: x over the 16-byte vectors of one token's row, y over tokens t0 + blockIdx.y
  constexpr int V = Vec16<T>::N;
  const int row_vecs = (H + 2 * G) * D / V;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= row_vecs) return;
  const int col = c * V;
  const int head = col / D, e = col % D;
  const int t = t0 + blockIdx.y;
  const int b = t / S, s = t % S, p = start_pos + s;
  const T *src = qkv + (size_t)t * (H + 2 * G) * D + col;
  Vec16<T> x = load16(src);
  if (head >= H + G) {
    const int g = head - H - G;
    store16(vc + (((size_t)b * G + g) * cache_seq + p) * D + e, x);
    return;
  }
  T *dst = head < H ? q_out + (size_t)t * H * D + head * D
                    : kc + (((size_t)b * G + (head - H)) * cache_seq + p) * D;
  if (!halves) {
    // pairs (e + 2k, e + 2k + 1) rotate by table[p][e/2 + k]; e/2 is a multiple of V/2,
    // so the cos/sin pairs load as 16-byte vectors
    const float4 *cs = reinterpret_cast<const float4 *>(table + (size_t)p * (D / 2) + e / 2);
    Vec16<T> o;
#pragma unroll
    for (int k = 0; k < V / 4; ++k) {
      const float4 c4 = cs[k];
      float a = x.get(4 * k), bb = x.get(4 * k + 1);
      o.set(4 * k, a * c4.x - bb * c4.y);
      o.set(4 * k + 1, a * c4.y + bb * c4.x);
      a = x.get(4 * k + 2);
      bb = x.get(4 * k + 3);
      o.set(4 * k + 2, a * c4.z - bb * c4.w);
      o.set(4 * k + 3, a * c4.w + bb * c4.z);
    }
    store16(dst + e, o);
  } else if (e < D / 2) {
    const float2 *cs = table + (size_t)p * (D / 2) + e;
    Vec16<T> y = load16(src + D / 2);
    Vec16<T> lo, hi;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float2 cv = cs[k];
      const float a = x.get(k), bb = y.get(k);
      lo.set(k, a * cv.x - bb * cv.y);
      hi.set(k, a * cv.y + bb * cv.x);
    }
    store16(dst + e, lo);
    store16(dst + e + D / 2, hi);
  }
}

template <typename T>
cudaError_t launch_rope_kv(const T *qkv, T *q_out, T *kc, T *vc, const float2 *table, int B, int S,
                           int start_pos, int H, int G, int D, int cache_seq, int halves, cudaStream_t st) {
  constexpr int V = Vec16<T>::N;
  const int ntok = B * S;
  const int row_vecs = (H + 2 * G) * D / V;
  if (ntok <= 0 || row_vecs <= 0) return cudaSuccess;
  if (halves && (D / 2) % V != 0) return cudaErrorInvalidValue;
  if (D % V != 0 || (D / 2) % (V / 2) != 0) return cudaErrorInvalidValue;
  const int threads = 256;
  const unsigned gx = (unsigned)((row_vecs + threads - 1) / threads);
  for (int t0 = 0; t0 < ntok; t0 += 65535) {  // grid y is at most 65535 tokens per launch
    const int n = ntok - t0 < 65535 ? ntok - t0 : 65535;
    count_launch();
    rope_kv_kernel<T><<<dim3(gx, (unsigned)n), threads, 0, st>>>(qkv, q_out, kc, vc, table, t0, S, start_pos, H, G,
                                                                 D, cache_seq, halves);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ------------------------------------------------------ SIMT attention ---
// "The Evolving Transformer 04 · LLaMA", §05 GQA: softmax(q k^T / sqrt(D)) v
// with query head h reading KV head h / (H / G) and keys j <= start_pos + s.
// One warp per (token, head); lanes split the head dimension; online softmax.
template <typename T>
__global__ void attention_simt_kernel(const T *__restrict__ q, const T *__restrict__ kc, const T *__restrict__ vc,
                                      T *__restrict__ o, int ntok, int S, int start_pos, int H, int G, int D,
                                      int cache_seq, float scale) {
  const size_t wid = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (size_t)ntok * H) return;
  const int t = (int)(wid / H), h = (int)(wid % H);
  const int b = t / S, s = t % S;
  const int g = h / (H / G);
  const int L = start_pos + s + 1;
  constexpr int MAXE = 4;  // D <= 128
  float qv[MAXE], acc[MAXE];
#pragma unroll
  for (int k = 0; k < MAXE; ++k) {
    const int e = lane + 32 * k;
    qv[k] = e < D ? to_f32<T>(q[((size_t)t * H + h) * D + e]) * scale : 0.f;
    acc[k] = 0.f;
  }
  const T *kb = kc + ((size_t)b * G + g) * cache_seq * D;
  const T *vb = vc + ((size_t)b * G + g) * cache_seq * D;
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < L; ++j) {
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < MAXE; ++k) {
      const int e = lane + 32 * k;
      if (e < D) dot = fmaf(qv[k], to_f32<T>(kb[(size_t)j * D + e]), dot);
    }
    dot = warp_sum(dot);
    const float mn = fmaxf(m, dot);
    const float corr = expf(m - mn);
    const float p = expf(dot - mn);
    l = l * corr + p;
#pragma unroll
    for (int k = 0; k < MAXE; ++k) {
      const int e = lane + 32 * k;
      if (e < D) acc[k] = fmaf(p, to_f32<T>(vb[(size_t)j * D + e]), acc[k] * corr);
    }
    m = mn;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < MAXE; ++k) {
    const int e = lane + 32 * k;
    if (e < D) o[((size_t)t * H + h) * D + e] = from_f32<T>(acc[k] * inv);
  }
}

template <typename T>
cudaError_t launch_attention_simt(const T *q, const T *kc, const T *vc, T *o, int B, int S, int start_pos, int H,
                                  int G, int D, int cache_seq, cudaStream_t st) {
  const size_t warps = (size_t)B * S * H;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((warps * 32 + threads - 1) / threads);
  count_launch();
  attention_simt_kernel<T><<<blocks, threads, 0, st>>>(q, kc, vc, o, B * S, S, start_pos, H, G, D, cache_seq,
                                                       1.0f / sqrtf((float)D));
  return cudaGetLastError();
}

// ------------------------------------------------------------ embedding ---
// "The Evolving Transformer 04 · LLaMA", §01 Embeddings: x = wte(ids), no position table.
template <typename T>
__global__ void embed_kernel(const int32_t *__restrict__ tokens, const T *__restrict__ E, T *__restrict__ x,
                             int ntok, int d, int vocab, int *status) {
  constexpr int V = Vec16<T>::N;
  const int nv = d / V;
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)ntok * nv) return;
  const int t = (int)(idx / nv), c = (int)(idx % nv) * V;
  const int id = tokens[t];
  Vec16<T> v;
  if (id < 0 || id >= vocab) {
    v.raw = make_uint4(0, 0, 0, 0);
    if (c == 0) report_status(status, DEV_BAD_TOKEN);
  } else {
    v = load16(E + (size_t)id * d + c);
  }
  store16(x + (size_t)t * d + c, v);
}

template <typename T>
cudaError_t launch_embed(const int32_t *tokens, const T *E, T *x, int ntok, int d, int vocab, int *status,
                         cudaStream_t st) {
  constexpr int V = Vec16<T>::N;
  const size_t total = (size_t)ntok * (d / V);
  if (total == 0) return cudaSuccess;
  count_launch();
  embed_kernel<T><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(tokens, E, x, ntok, d, vocab, status);
  return cudaGetLastError();
}

// ------------------------------------------------------- greedy decoding ---
// Row r of the logits picks the id of its maximum; among equal maxima the
// lowest id wins, and NaN is never picked (a row of NaN gives id 0).
__device__ __forceinline__ void argmax_merge(float &v, int &i, float ov, int oi) {
  if (ov > v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

__global__ void argmax_rows_kernel(const float *__restrict__ logits, int vocab, int32_t *__restrict__ out,
                                   int out_stride, int32_t *__restrict__ next) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const float *l = logits + (size_t)blockIdx.x * vocab;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int j = threadIdx.x; j < vocab; j += blockDim.x) argmax_merge(best, bi, __ldcs(l + j), j);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    argmax_merge(best, bi, ov, oi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (lane == 0) {
    sv[warp] = best;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    best = lane < nwarps ? sv[lane] : -INFINITY;
    bi = lane < nwarps ? si[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(best, bi, ov, oi);
    }
    if (lane == 0) {
      const int id = bi == INT_MAX ? 0 : bi;
      out[(size_t)blockIdx.x * out_stride] = id;
      if (next != nullptr) next[blockIdx.x] = id;
    }
  }
}

cudaError_t launch_argmax_rows(const float *logits, int rows, int vocab, int32_t *out, int out_stride, int32_t *next,
                               cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  count_launch();
  argmax_rows_kernel<<<rows, 1024, 0, st>>>(logits, vocab, out, out_stride, next);
  return cudaGetLastError();
}

// out[b] = x[b][S - 1] for rows of width d (the last position of each sequence).
template <typename T>
__global__ void gather_last_rows_kernel(const T *__restrict__ x, T *__restrict__ out, int B, int S, int d) {
  constexpr int V = Vec16<T>::N;
  const int nv = d / V;
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)B * nv) return;
  const int b = (int)(idx / nv), c = (int)(idx % nv) * V;
  store16(out + (size_t)b * d + c, load16(x + ((size_t)b * S + S - 1) * d + c));
}

template <typename T>
cudaError_t launch_gather_last_rows(const T *x, T *out, int B, int S, int d, cudaStream_t st) {
  constexpr int V = Vec16<T>::N;
  const size_t total = (size_t)B * (d / V);
  if (total == 0) return cudaSuccess;
  count_launch();
  gather_last_rows_kernel<T><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(x, out, B, S, d);
  return cudaGetLastError();
}

#define INSTANTIATE(T)                                                                                            \
  template cudaError_t launch_rmsnorm<T>(const T *, const T *, T *, int, int, float, cudaStream_t);               \
  template cudaError_t launch_gemm_simt<T>(const T *, const T *, const T *, const T *, void *, int, int, int, int, \
                                           cudaStream_t);                                                         \
  template cudaError_t launch_rope_kv<T>(const T *, T *, T *, T *, const float2 *, int, int, int, int, int, int,  \
                                         int, int, cudaStream_t);                                                 \
  template cudaError_t launch_attention_simt<T>(const T *, const T *, const T *, T *, int, int, int, int, int,    \
                                                int, int, cudaStream_t);                                          \
  template cudaError_t launch_embed<T>(const int32_t *, const T *, T *, int, int, int, int *, cudaStream_t);    \
  template cudaError_t launch_gather_last_rows<T>(const T *, T *, int, int, int, cudaStream_t);

INSTANTIATE(float)
INSTANTIATE(bf16)

}  // namespace llama
