// Decode-step attention (S = 1) over the bf16 KV cache: memory-bound split-KV.
// "Full Llama 3 transformer block", How it works (cache read up to start_pos);
// "Llama 4 From Scratch", Worked example (the KV cache is what limits
// long-context inference: each cached byte is read once per step here).
//
// CTA = (sequence b, KV head g, chunk of 256 cached positions); 8 warps.
//   * The chunk streams through a 3-stage shared-memory ring of 64-position
//     K and V sub-tiles, each one contiguous 1-D bulk async copy.
//   * All r = H/G query heads of group g are served by the same K/V bytes:
//     lane (key, head) of a warp computes one q.k dot product (q pre-scaled by
//     log2(e)/sqrt(D), fp32), each warp keeps an online softmax per head over
//     its 8 positions of every sub-tile, and accumulates o[head][d] for its
//     d-slice of every head.
//   * At the end the 8 warps merge (log-sum-exp) and the CTA writes an fp32
//     partial (o, m, l) per head -- or, with one chunk, the normalised output.
//   * A combine kernel merges the chunks' partials per (b, h).
#include <cmath>
#include <mutex>

#include "decode_combine.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {
namespace {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int DEC_SUB = 64;          // positions per stage (8 per warp)
constexpr int DEC_KW = DEC_SUB / DEC_WARPS;
constexpr int DEC_CHUNK = 256;       // positions per CTA
constexpr int DEC_STAGES = 3;

template <int D, int RP>
struct DecLayout {
  static constexpr int ROW = D * 2;                       // bytes per cached position
  static constexpr int STAGE = 2 * DEC_SUB * ROW;         // K then V
  static constexpr int OFF_Q = DEC_STAGES * STAGE;        // fp32 q [RP][D + 4]
  static constexpr int QROW = D + 4;
  static constexpr int OFF_P = OFF_Q + RP * QROW * 4;     // per warp [DEC_KW][RP] fp32
  static constexpr int OFF_BAR = OFF_P + DEC_WARPS * DEC_KW * RP * 4;
  static constexpr int BYTES = 16 + OFF_BAR + 2 * DEC_STAGES * 8;
  static constexpr int EPL = D / 32;                      // d elements per lane
  static constexpr int DOTS = (DEC_KW * RP + 31) / 32;    // (position, head) dot products per lane
};

struct DecArgs {
  const bf16 *q;
  const bf16 *kc, *vc;
  bf16 *o;
  float *part;  // [B][H][n_split][D + 2]: o (unnormalised), m, l
  int H, G, r, cache_seq, kv_len, n_split;
  float scale_log2;
  int *status;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int D, int RP>
__global__ void __launch_bounds__(DEC_THREADS) attn_decode_kernel(DecArgs a) {
  using L = DecLayout<D, RP>;
  extern __shared__ __align__(16) uint8_t smem[];
  float *qs = reinterpret_cast<float *>(smem + L::OFF_Q);
  float *pbuf_all = reinterpret_cast<float *>(smem + L::OFF_P);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  const uint32_t s0 = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (DEC_STAGES + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int k0 = split * DEC_CHUNK;
  const int k1 = min(a.kv_len, k0 + DEC_CHUNK);
  const int n_sub = (k1 - k0 + DEC_SUB - 1) / DEC_SUB;
  const size_t head_base = ((size_t)b * a.G + g) * a.cache_seq;
  const bf16 *kg = a.kc + (head_base + k0) * D;
  const bf16 *vg = a.vc + (head_base + k0) * D;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DEC_STAGES; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), DEC_WARPS);
    }
    ptx::fence_mbar_init();
  }
  // q of the group's heads, pre-scaled, fp32; head slots >= r are zero.
  for (int i = threadIdx.x; i < RP * D; i += DEC_THREADS) {
    const int hh = i / D, d = i % D;
    float v = 0.f;
    if (hh < a.r) v = __bfloat162float(a.q[((size_t)b * a.H + g * a.r + hh) * D + d]) * a.scale_log2;
    qs[hh * L::QROW + d] = v;
  }
  __syncthreads();

  auto issue = [&](int j) {
    const int s = j % DEC_STAGES;
    const int keys = min(DEC_SUB, k1 - k0 - j * DEC_SUB);
    const uint32_t bytes = (uint32_t)keys * L::ROW;
    ptx::mbar_arrive_expect_tx(full(s), 2 * bytes);
    const uint64_t once = ptx::policy_evict_first();  // each cached key is read once per step
    ptx::bulk_load_hint(s0 + s * L::STAGE, kg + (size_t)j * DEC_SUB * D, bytes, full(s), once);
    ptx::bulk_load_hint(s0 + s * L::STAGE + DEC_SUB * L::ROW, vg + (size_t)j * DEC_SUB * D, bytes, full(s), once);
  };
  volatile int abort_local = 0;
  int issued = 0;  // thread 0: sub-tiles whose copies have been issued
  if (threadIdx.x == 0)
    for (; issued < min(DEC_STAGES, n_sub); ++issued) issue(issued);

  float m_h = -INFINITY, l_h = 0.f;  // softmax state of this lane's head (lane % RP)
  float o[RP][L::EPL];
#pragma unroll
  for (int h = 0; h < RP; ++h)
#pragma unroll
    for (int e = 0; e < L::EPL; ++e) o[h][e] = 0.f;
  float *pbuf = pbuf_all + warp * DEC_KW * RP;
  bool ok = true;

  for (int j = 0; j < n_sub; ++j) {
    const int s = j % DEC_STAGES;
    ok = ptx::mbar_wait(full(s), (j / DEC_STAGES) & 1, &abort_local, a.status, DEV_TIMEOUT_ATTN);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint8_t *ks = smem + s * L::STAGE;
    const uint8_t *vs = ks + DEC_SUB * L::ROW;
    const int kbase = j * DEC_SUB + warp * DEC_KW;  // chunk-relative first position of this warp
    const int nvalid = max(0, min(DEC_KW, (k1 - k0) - kbase));
    // scores: lane pair index -> (position, head)
    float sc[L::DOTS];
#pragma unroll
    for (int i = 0; i < L::DOTS; ++i) {
      const int idx = lane + 32 * i;
      const int kl = idx / RP, hd = idx % RP;
      float acc = -INFINITY;
      if (idx < DEC_KW * RP && kl < nvalid) {
        const uint8_t *krow = ks + (size_t)(warp * DEC_KW + kl) * L::ROW;
        const float *qrow = qs + hd * L::QROW;
        acc = 0.f;
#pragma unroll
        for (int c = 0; c < L::ROW / 16; ++c) {
          const int cc = (c + kl) & (L::ROW / 16 - 1);  // rotate chunks: no bank conflicts between rows
          float kf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(krow + cc * 16), kf);
          const float4 q0 = *reinterpret_cast<const float4 *>(qrow + cc * 8);
          const float4 q1 = *reinterpret_cast<const float4 *>(qrow + cc * 8 + 4);
          acc = fmaf(kf[0], q0.x, acc);
          acc = fmaf(kf[1], q0.y, acc);
          acc = fmaf(kf[2], q0.z, acc);
          acc = fmaf(kf[3], q0.w, acc);
          acc = fmaf(kf[4], q1.x, acc);
          acc = fmaf(kf[5], q1.y, acc);
          acc = fmaf(kf[6], q1.z, acc);
          acc = fmaf(kf[7], q1.w, acc);
        }
      }
      sc[i] = acc;
    }
    // tile max per head over the warp's positions (lanes sharing lane % RP)
    float mt = sc[0];
#pragma unroll
    for (int i = 1; i < L::DOTS; ++i) mt = fmaxf(mt, sc[i]);
#pragma unroll
    for (int off = RP; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float m_new = fmaxf(m_h, mt);
    const float alpha = (m_new == -INFINITY) ? 1.f : ptx::ex2_approx(m_h - m_new);
    float psum = 0.f;
#pragma unroll
    for (int i = 0; i < L::DOTS; ++i) {
      const int idx = lane + 32 * i;
      const float p = (sc[i] == -INFINITY) ? 0.f : ptx::ex2_approx(sc[i] - m_new);
      psum += p;
      if (idx < DEC_KW * RP) pbuf[idx] = p;  // pbuf[position][head]
    }
#pragma unroll
    for (int off = RP; off < 32; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l_h = l_h * alpha + psum;
    m_h = m_new;
    __syncwarp();
    // rescale every head's accumulator, then o[h][d] += sum_k p[k][h] v[k][d]
#pragma unroll
    for (int h = 0; h < RP; ++h) {
      const float ah = __shfl_sync(0xffffffffu, alpha, h);
#pragma unroll
      for (int e = 0; e < L::EPL; ++e) o[h][e] *= ah;
    }
    for (int kl = 0; kl < nvalid; ++kl) {
      const uint8_t *vrow = vs + (size_t)(warp * DEC_KW + kl) * L::ROW + lane * L::EPL * 2;
      float vf[L::EPL];
      if constexpr (L::EPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(vrow);
        vf[0] = __uint_as_float(u.x << 16);
        vf[1] = __uint_as_float(u.x & 0xFFFF0000u);
        vf[2] = __uint_as_float(u.y << 16);
        vf[3] = __uint_as_float(u.y & 0xFFFF0000u);
      } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(vrow);
        vf[0] = __uint_as_float(u << 16);
        vf[1] = __uint_as_float(u & 0xFFFF0000u);
      }
#pragma unroll
      for (int h = 0; h < RP; ++h) {
        const float p = pbuf[kl * RP + h];
#pragma unroll
        for (int e = 0; e < L::EPL; ++e) o[h][e] = fmaf(p, vf[e], o[h][e]);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty(s));
    // refill this stage with sub-tile j + DEC_STAGES once every warp released it
    if (threadIdx.x == 0 && j + DEC_STAGES < n_sub) {
      if (ptx::mbar_wait(empty(s), (j / DEC_STAGES) & 1, &abort_local, a.status, DEV_TIMEOUT_PRODUCER)) {
        issue(j + DEC_STAGES);
        ++issued;
      }
    }
  }
  // A consumer whose wait gave up leaves copies in flight: they land before the
  // stage buffers are reused below (or the CTA exits).  Sub-tile j + DEC_STAGES
  // is issued only once every warp has consumed sub-tile j, so only the last
  // DEC_STAGES issued copies can still be outstanding.
  if (threadIdx.x == 0)
    for (int j = max(0, issued - DEC_STAGES); j < issued; ++j)
      ptx::mbar_drain(full(j % DEC_STAGES), (j / DEC_STAGES) & 1, a.status, DEV_TIMEOUT_ATTN);
  __syncthreads();
  // ------------------------------------------------------------- merge ---
  // Reuse the stage buffers: per warp [RP][D] o, then [RP] m and l.
  float *mo = reinterpret_cast<float *>(smem);
  float *mm = mo + DEC_WARPS * RP * D;
  float *ml = mm + DEC_WARPS * RP;
#pragma unroll
  for (int h = 0; h < RP; ++h)
#pragma unroll
    for (int e = 0; e < L::EPL; ++e) mo[(warp * RP + h) * D + lane * L::EPL + e] = o[h][e];
  if (lane < RP) {
    mm[warp * RP + lane] = m_h;
    ml[warp * RP + lane] = l_h;
  }
  __syncthreads();
  if (!ok) return;
  for (int i = threadIdx.x; i < RP * D; i += DEC_THREADS) {
    const int h = i / D, d = i % D;
    if (h >= a.r) continue;
    float m = -INFINITY;
    for (int w = 0; w < DEC_WARPS; ++w) m = fmaxf(m, mm[w * RP + h]);
    float ov = 0.f, lv = 0.f;
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float mw = mm[w * RP + h];
      const float f = (mw == -INFINITY) ? 0.f : ptx::ex2_approx(mw - m);
      ov = fmaf(f, mo[(w * RP + h) * D + d], ov);
      lv = fmaf(f, ml[w * RP + h], lv);
    }
    const int hq = g * a.r + h;
    if (a.n_split == 1) {
      a.o[((size_t)b * a.H + hq) * D + d] = __float2bfloat16_rn(ov / lv);
    } else {
      float *pp = a.part + (((size_t)b * a.H + hq) * a.n_split + split) * (D + 2);
      pp[d] = ov;
      if (d == 0) {
        pp[D] = m;
        pp[D + 1] = lv;
      }
    }
  }
}

// Merge the n_split chunk partials of every (b, h): one CTA of D threads each.
template <int D>
__global__ void __launch_bounds__(D) attn_decode_combine(const float *__restrict__ part, bf16 *__restrict__ o, int H,
                                                         int n_split) {
  allow_dependents_launch();
  grid_dependency_wait();
  decode_combine_element<D>(part, o, blockIdx.x, threadIdx.x, n_split);
}

template <int D, int RP>
cudaError_t launch_dec(const DecArgs &base, int B, const AttnScratch &scratch, cudaStream_t st) {
  using L = DecLayout<D, RP>;
  static PerContextOnce attr;
  const cudaError_t attr_err = attr.run([] {
    return cudaFuncSetAttribute(attn_decode_kernel<D, RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const size_t per_seq = (size_t)base.H * base.n_split * (D + 2) * sizeof(float);
  int group = base.n_split == 1 ? B : (int)(scratch.bytes / per_seq);
  if (group < 1) return cudaErrorMemoryAllocation;
  if (group > 65535) group = 65535;
  for (int b0 = 0; b0 < B; b0 += group) {
    const int nb = min(group, B - b0);
    DecArgs a = base;
    a.q = base.q + (size_t)b0 * base.H * D;
    a.kc = base.kc + (size_t)b0 * base.G * base.cache_seq * D;
    a.vc = base.vc + (size_t)b0 * base.G * base.cache_seq * D;
    a.o = base.o + (size_t)b0 * base.H * D;
    dim3 grid(base.n_split, base.G, nb);
    count_launch();
    attn_decode_kernel<D, RP><<<grid, DEC_THREADS, L::BYTES, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (base.n_split > 1) {
      count_launch();
      attn_decode_combine<D><<<nb * base.H, D, 0, st>>>(a.part, a.o, base.H, base.n_split);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

template <int D>
cudaError_t dispatch_rp(const DecArgs &a, int B, int rp, const AttnScratch &scratch, cudaStream_t st) {
  switch (rp) {
    case 1: return launch_dec<D, 1>(a, B, scratch, st);
    case 2: return launch_dec<D, 2>(a, B, scratch, st);
    case 4: return launch_dec<D, 4>(a, B, scratch, st);
    case 8: return launch_dec<D, 8>(a, B, scratch, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

size_t attn_decode_scratch_bytes(int max_tokens, int H, int D, int max_seq) {
  const size_t n_split = (size_t)((max_seq + DEC_CHUNK - 1) / DEC_CHUNK);
  const size_t want = (size_t)max_tokens * H * n_split * (D + 2) * sizeof(float);
  const size_t cap = (size_t)64 << 20;  // larger batches are processed in groups
  const size_t one = (size_t)H * n_split * (D + 2) * sizeof(float);
  return want < cap ? want : (one > cap ? one : cap);
}

cudaError_t launch_decode_combine(const float *part, bf16 *o, int BH, int D, int n_split, cudaStream_t st) {
  if (D == 128) {
    count_launch();
    return launch_pdl(attn_decode_combine<128>, dim3(BH), dim3(128), 0, st, part, o, 0, n_split);
  } else if (D == 64) {
    count_launch();
    return launch_pdl(attn_decode_combine<64>, dim3(BH), dim3(64), 0, st, part, o, 0, n_split);
  }
  return cudaErrorInvalidValue;
}

bool attn_decode_supported(int H, int G, int D) {
  const int r = H / G;
  return (D == 64 || D == 128) && r <= 8;
}

cudaError_t launch_attn_decode(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos, int H,
                               int G, int D, int cache_seq, const AttnScratch &scratch, int *status,
                               cudaStream_t st) {
  const int r = H / G;
  int rp = 1;
  while (rp < r) rp *= 2;
  DecArgs a;
  a.q = q;
  a.kc = kc;
  a.vc = vc;
  a.o = o;
  a.part = reinterpret_cast<float *>(scratch.partial);
  a.H = H;
  a.G = G;
  a.r = r;
  a.cache_seq = cache_seq;
  a.kv_len = start_pos + 1;
  a.n_split = (a.kv_len + DEC_CHUNK - 1) / DEC_CHUNK;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  a.status = status;
  if (a.n_split > 1 && scratch.partial == nullptr) return cudaErrorInvalidValue;
  if (D == 128) return dispatch_rp<128>(a, B, rp, scratch, st);
  if (D == 64) return dispatch_rp<64>(a, B, rp, scratch, st);
  return cudaErrorInvalidValue;
}

}  // namespace llama
