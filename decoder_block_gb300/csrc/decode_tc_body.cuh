// Tensor-core decode attention body, shared by its own kernel (decode_tc.cu)
// and the fused decode-step kernel (decode_fused.cu).
//
// Decode-step attention (S = 1, d_head = 128) on tcgen05 tensor cores.
// "Full Llama 3 transformer block", How it works (cached keys 0 .. start_pos);
// "The Evolving Transformer 04 · LLaMA", §05 GQA (head h reads KV head h / r).
//
// The step is HBM-bound (every cached K/V byte is read once); the tensor cores
// only keep the CUDA cores free so that the loads, not the instruction issue,
// set the pace.  Swap-AB form per 128-position tile of one (b, g):
//   S^T[128 positions x 16] = K_tile . Q_g^T       (M = positions, N = the group's
//                                                   query heads padded to 16)
//   O^T[128 d x 16]        += V_tile^T . P^T       (V read as an MN-major operand)
// Persistent CTAs (one per SM) walk work items (b, g, chunk of 512 positions):
//   warp 0      TMA producer: takes the next work item (from a grid-wide
//               counter, so CTAs that stream faster take more items; or a
//               fixed share), passes its index to the other roles next to its
//               Q buffer (-1: no more), loads Q_g (16 rows) and the K and V
//               tiles into a 3-stage ring (tensor maps end at start_pos + 1:
//               zeros beyond);
//   warp 1      tcgen05.mma issuer (double-buffered S^T, O^T per item parity);
//   warps 2-5   one thread per position (TMEM lane): per-head max over the
//               tile (warp shuffles + shared memory), p = 2^(s*log2e/sqrt(D) - m)
//               written as bf16 P^T into shared memory, lazy O rescale, and at
//               item end the fp32 partial (o, m, l) per head for the combine step.
#pragma once

#include <cuda.h>

#include "kernels.h"
#include "phase_sync.cuh"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {

constexpr int DT_D = 128;
constexpr int DT_TILE = 128;     // positions per tile
constexpr int DT_CHUNK = 512;    // positions per work item
constexpr int DT_STAGES = 3;
constexpr int DT_N = 16;         // query-head columns (r <= 16)
constexpr int DT_THREADS = 192;
constexpr float DT_RESCALE = 8.0f;

struct DtLayout {
  static constexpr int ATOM = DT_TILE * 128;           // 128 rows x 128 bytes
  static constexpr int KV_BYTES = 2 * ATOM;             // 128 positions x 128 d x 2 B
  static constexpr int Q_BYTES = 2 * DT_N * 128;        // 16 rows, two 64-column atoms
  static constexpr int P_BYTES = 2 * DT_N * 128;        // 16 rows x 128 positions, two atoms
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + DT_STAGES * KV_BYTES;
  static constexpr int OFF_Q = OFF_V + DT_STAGES * KV_BYTES;  // 2 buffers
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;           // 2 buffers
  static constexpr int OFF_RED = OFF_P + 2 * P_BYTES;          // [3 sets][4 warps][DT_N] floats
  static constexpr int OFF_ITEM = OFF_RED + 3 * 4 * DT_N * 4;  // work item of each Q buffer (-1: no more)
  static constexpr int OFF_BAR = OFF_ITEM + 16;
  // kv_full[3], kv_empty[3], q_full[2], q_empty[2], s_full[2], p_full[2], p_free[2], o_full[2], o_free[2], fin,
  // red_full[2] (per-tile max exchange), lred_full (per-item sum exchange)
  static constexpr int NBAR = 2 * DT_STAGES + 14 + 1 + 3;
  static constexpr int BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 64;  // S^T x2 (16 each) + O^T x2 (16 each)
};

struct DtArgs {
  float *part;  // [B][H][n_split][D + 2]
  bf16 *o;      // [B][H][D] when n_split == 1
  int B, H, G, r, kv_len, n_split, n_items;
  float scale_log2;
  int *status;
  int *items;  // [0] next work item, [1] CTAs finished (zero at launch, left zero); null: fixed share
};

// The 4 softmax warps exchange per-head values through shared memory; each
// exchange is one mbarrier phase (one arrival per warp) waited on with the
// same bounded wait as every other barrier, so a warp that gives up can never
// leave the others blocked.
template <int N>
__device__ __forceinline__ bool exchange(float *slot_row, const float (&v)[N], uint32_t bar, uint32_t parity,
                                         volatile int *abort, int *status) {
  const int lane = threadIdx.x & 31;
  if (lane < N) {
    float x = v[0];
#pragma unroll
    for (int h = 1; h < N; ++h)
      if (lane == h) x = v[h];
    slot_row[lane] = x;
  }
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(bar);
  const bool ok = ptx::mbar_wait(bar, parity, abort, status, DEV_TIMEOUT_ATTN);
  return __all_sync(0xffffffffu, ok);
}

// RN: head columns the softmax works on (the smallest of 4, 8, 16 that is >= r);
// P^T rows RN .. 15 stay zero, so the MMAs' padded columns contribute nothing.
template <int RN>
__device__ __forceinline__ void attn_decode_tc_run(const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                                   const CUtensorMap *tmV, const DtArgs &a, const PhaseSync sync) {
  using L = DtLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *red = reinterpret_cast<float *>(smem + L::OFF_RED);
  volatile int *item_slot = reinterpret_cast<volatile int *>(smem + L::OFF_ITEM);

  const uint32_t s0 = ptx::smem_u32(smem);
  const uint32_t b0 = ptx::smem_u32(bars);
  auto kv_full = [&](int s) { return b0 + 8u * s; };
  auto kv_empty = [&](int s) { return b0 + 8u * (DT_STAGES + s); };
  auto q_full = [&](int i) { return b0 + 8u * (2 * DT_STAGES + i); };
  auto q_empty = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 2 + i); };
  auto s_full = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 4 + i); };
  auto p_full = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 6 + i); };
  auto p_free = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 8 + i); };
  auto o_full = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 10 + i); };
  auto o_free = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 12 + i); };
  const uint32_t fin = b0 + 8u * (2 * DT_STAGES + 14);
  auto red_full = [&](int i) { return b0 + 8u * (2 * DT_STAGES + 15 + i); };
  const uint32_t lred_full = b0 + 8u * (2 * DT_STAGES + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < DT_STAGES; ++s) {
      ptx::mbar_init(kv_full(s), 1);
      ptx::mbar_init(kv_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(q_full(i), 1);
      ptx::mbar_init(q_empty(i), 1);
      ptx::mbar_init(s_full(i), 1);
      ptx::mbar_init(p_full(i), 128);
      ptx::mbar_init(p_free(i), 1);
      ptx::mbar_init(o_full(i), 1);
      ptx::mbar_init(o_free(i), 128);
    }
    ptx::mbar_init(fin, 1);
    ptx::mbar_init(red_full(0), 4);
    ptx::mbar_init(red_full(1), 4);
    ptx::mbar_init(lred_full, 4);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1 && !sync.fused()) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sync.fused() ? sync.tmem : *tmem_slot;
  // q and the cache come from earlier kernels (programmatic dependent launch)
  // or from the previous phase of the fused kernel
  bool go = true;
  if (!sync.fused()) {
    allow_dependents_launch();
    grid_dependency_wait();
  } else {
    if (threadIdx.x == 0 && !phase_wait(sync, a.status)) *abort_flag = 1;
    __syncthreads();
    go = *abort_flag == 0;
  }

  // Work item -> (b, g, chunk).
  auto item_coords = [&](int it, int &b, int &g, int &k0, int &nt) {
    const int split = it % a.n_split;
    const int bg = it / a.n_split;
    b = bg / a.G;
    g = bg % a.G;
    k0 = split * DT_CHUNK;
    const int k1 = min(a.kv_len, k0 + DT_CHUNK);
    nt = (k1 - k0 + DT_TILE - 1) / DT_TILE;
  };

  if (!go) {
    // inputs never became ready: nothing was issued
  } else if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(tmQ);
      ptx::tma_prefetch_desc(tmK);
      ptx::tma_prefetch_desc(tmV);
      int tile = 0, nq = 0;
      bool ok = true;
      for (;; ++nq) {
        int it = a.items != nullptr ? atomicAdd(a.items, 1) : (int)blockIdx.x + nq * (int)gridDim.x;
        if (it >= a.n_items) it = -1;
        const int qi = nq & 1;
        if (!ptx::mbar_wait(q_empty(qi), ((nq >> 1) & 1) ^ 1, abort_flag, a.status, DEV_TIMEOUT_PRODUCER)) break;
        item_slot[qi] = it;  // published to the other roles by the q_full arrival
        if (it < 0) {
          ptx::mbar_arrive(q_full(qi));
          break;
        }
        int b, g, k0, nt;
        item_coords(it, b, g, k0, nt);
        ptx::mbar_arrive_expect_tx(q_full(qi), L::Q_BYTES);
        for (int at = 0; at < 2; ++at)
          ptx::tma_load_2d(s0 + L::OFF_Q + qi * L::Q_BYTES + at * (DT_N * 128), tmQ, at * 64, b * a.H + g * a.r,
                           q_full(qi));
        for (int j = 0; j < nt; ++j, ++tile) {
          const int st = tile % DT_STAGES;
          const uint32_t ph = (tile / DT_STAGES) & 1;
          if (!ptx::mbar_wait(kv_empty(st), ph ^ 1, abort_flag, a.status, DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(kv_full(st), 2 * L::KV_BYTES);
          const int key = k0 + j * DT_TILE;
          const uint64_t once = ptx::policy_evict_first();  // each cached key is read once per step
          for (int at = 0; at < 2; ++at) {
            ptx::tma_load_4d_hint(s0 + L::OFF_K + st * L::KV_BYTES + at * L::ATOM, tmK, at * 64, key, g, b,
                                  kv_full(st), once);
            ptx::tma_load_4d_hint(s0 + L::OFF_V + st * L::KV_BYTES + at * L::ATOM, tmV, at * 64, key, g, b,
                                  kv_full(st), once);
          }
        }
        if (!ok) {
          ++nq;
          break;
        }
      }
      // drain the last issued loads
      for (int t = max(0, tile - DT_STAGES); t < tile; ++t)
        ptx::mbar_drain(kv_full(t % DT_STAGES), (t / DT_STAGES) & 1, a.status, DEV_TIMEOUT_PRODUCER);
      if (nq > 0) ptx::mbar_drain(q_full((nq - 1) & 1), ((nq - 1) >> 1) & 1, a.status, DEV_TIMEOUT_PRODUCER);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(DT_TILE, DT_N, false);
      // O^T = V^T P^T: A = V^T (M = d, MN-major), B = P^T (N = heads, K-major)
      constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(DT_D, DT_N, false) | (1u << 15);
      int tile = 0, nq = 0;
      bool ok = true;
      for (; ok; ++nq) {
        const int qi = nq & 1, ob = nq & 1;
        if (!ptx::mbar_wait(q_full(qi), (nq >> 1) & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
        const int it = item_slot[qi];
        if (it < 0) break;  // no more work items
        int b, g, k0, nt;
        item_coords(it, b, g, k0, nt);
        if (!ptx::mbar_wait(o_free(ob), ((nq >> 1) & 1) ^ 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
        const uint32_t qbase = s0 + L::OFF_Q + qi * L::Q_BYTES;
        // S^T of tile t (global tile counter) into buffer t & 1, reading K stage t % STAGES.
        auto issue_s = [&](int t) -> bool {
          const int st = t % DT_STAGES;
          if (!ptx::mbar_wait(kv_full(st), (t / DT_STAGES) & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) return false;
          ptx::tc_fence_after();
          const uint32_t kb = s0 + L::OFF_K + st * L::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < DT_D / 16; ++kk) {
            const uint32_t ka = (kk / 4) * L::ATOM + (kk % 4) * 32;
            const uint32_t qa = (kk / 4) * (DT_N * 128) + (kk % 4) * 32;
            ptx::mma_bf16_ss(tmem + (t & 1) * DT_N, ptx::smem_desc_sw128(kb + ka), ptx::smem_desc_sw128(qbase + qa),
                             idesc_s, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(s_full(t & 1));
          return true;
        };
        ok = issue_s(tile);
        for (int j = 0; j < nt && ok; ++j, ++tile) {
          // one tile ahead: the softmax of this tile overlaps the next S^T
          if (j + 1 < nt && !issue_s(tile + 1)) {
            ok = false;
            break;
          }
          const int st = tile % DT_STAGES;
          const int sb = tile & 1;
          if (!ptx::mbar_wait(p_full(sb), (tile >> 1) & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t vb = s0 + L::OFF_V + st * L::KV_BYTES;
          const uint32_t pb = s0 + L::OFF_P + sb * L::P_BYTES;
#pragma unroll
          for (int kk = 0; kk < DT_TILE / 16; ++kk) {
            const uint64_t adesc = ptx::smem_desc_sw128_mn(vb + kk * 16 * 128, L::ATOM, 1024);
            const uint32_t pa = (kk / 4) * (DT_N * 128) + (kk % 4) * 32;
            ptx::mma_bf16_ss(tmem + 32 + ob * DT_N, adesc, ptx::smem_desc_sw128(pb + pa), idesc_o,
                             (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(p_free(sb));
          ptx::mma_commit(kv_empty(st));
        }
        if (!ok) break;
        ptx::mma_commit(q_empty(qi));
        ptx::mma_commit(o_full(ob));
      }
      ptx::mma_commit(fin);
      ptx::mbar_drain(fin, 0, a.status, DEV_TIMEOUT_MMA);
    }
  } else {
    // ------------------------------------------------- softmax / epilogue ---
    const int w4 = warp - 2;             // 0..3
    const int qq = warp & 3;             // TMEM lane quarter
    const int row = qq * 32 + lane;      // tile position (S^T) / d (O^T)
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    if (RN < DT_N) {  // P^T rows the softmax never writes: zero once for both buffers
      uint4 *pz = reinterpret_cast<uint4 *>(smem + L::OFF_P);
      for (int i = threadIdx.x - 64; i < 2 * L::P_BYTES / 16; i += 128) pz[i] = make_uint4(0, 0, 0, 0);
      ptx::fence_proxy_async_smem();
    }
    int tile = 0, nq = 0;
    bool ok = true;
    for (; ok; ++nq) {
      // the item of Q buffer nq & 1 (the producer's q_full arrival publishes it;
      // waiting here never runs ahead: that buffer is refilled only after this
      // item's last PV product, which needs this warp's P)
      ok = ptx::mbar_wait(q_full(nq & 1), (nq >> 1) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int it = item_slot[nq & 1];
      if (it < 0) break;  // no more work items
      int b, g, k0, nt;
      item_coords(it, b, g, k0, nt);
      const int ob = nq & 1;
      const int k1 = min(a.kv_len, k0 + DT_CHUNK);
      float m_run[RN], l_run[RN];
#pragma unroll
      for (int h = 0; h < RN; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
      for (int j = 0; j < nt; ++j, ++tile) {
        const int sb = tile & 1;
        ok = ptx::mbar_wait(s_full(sb), (tile >> 1) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        float s[DT_N];
        ptx::tmem_ld16(lane_base + sb * DT_N, s);
        ptx::tmem_ld_wait();
        const bool valid = k0 + j * DT_TILE + row < k1;
        // per-head tile max over the 128 positions: warp shuffles, then across the 4 warps
        float mx[RN];
#pragma unroll
        for (int h = 0; h < RN; ++h) {
          float v = (valid && h < a.r) ? s[h] : -INFINITY;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
          mx[h] = v;
        }
        float *rs = red + (tile & 1) * (4 * DT_N);
        if (!exchange(rs + w4 * DT_N, mx, red_full(tile & 1), (tile >> 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        bool need_any = false;
        float alpha[RN];
#pragma unroll
        for (int h = 0; h < RN; ++h) {
          const float t = fmaxf(fmaxf(rs[h], rs[DT_N + h]), fmaxf(rs[2 * DT_N + h], rs[3 * DT_N + h]));
          const float mt = t * a.scale_log2;
          alpha[h] = 1.f;
          if (h < a.r && mt > m_run[h] + DT_RESCALE) {
            alpha[h] = ptx::ex2_approx(m_run[h] - mt);
            m_run[h] = mt;
            need_any = true;
          }
        }
        // P^T into shared memory: row h (query head), column = position, 128-byte swizzle
        ok = ptx::mbar_wait(p_free(sb), ((tile >> 1) & 1) ^ 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        uint8_t *pbuf = smem + L::OFF_P + sb * L::P_BYTES + (row / 64) * (DT_N * 128);
        const int c = row % 64;
#pragma unroll
        for (int h = 0; h < RN; ++h) {
          const float p = (valid && h < a.r) ? ptx::ex2_approx(fmaf(s[h], a.scale_log2, -m_run[h])) : 0.f;
          l_run[h] = l_run[h] * alpha[h] + p;
          const int chunk = (c >> 3) ^ (h & 7);
          *reinterpret_cast<bf16 *>(pbuf + h * 128 + chunk * 16 + (c & 7) * 2) = __float2bfloat16_rn(p);
        }
        // lazy rescale of the running O^T (thread = d row) before this tile's PV is issued
        if (need_any && j > 0) {
          ok = ptx::mbar_wait(p_free(sb ^ 1), (((tile - 1) >> 1) & 1), abort_flag, a.status, DEV_TIMEOUT_ATTN);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          float ov[DT_N];
          ptx::tmem_ld16(lane_base + 32 + ob * DT_N, ov);
          ptx::tmem_ld_wait();
          uint32_t wv[DT_N];
#pragma unroll
          for (int h = 0; h < DT_N; ++h) wv[h] = __float_as_uint(h < RN ? ov[h] * alpha[h < RN ? h : 0] : ov[h]);
          ptx::tmem_st16(lane_base + 32 + ob * DT_N, wv);
          ptx::tmem_st_wait();
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full(sb));
      }
      if (!ok) break;
      // item end: reduce l over the 128 positions, read O^T, write the partial
      ok = ptx::mbar_wait(o_full(ob), (nq >> 1) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float ov[DT_N];
      ptx::tmem_ld16(lane_base + 32 + ob * DT_N, ov);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(o_free(ob));
#pragma unroll
      for (int h = 0; h < RN; ++h) {
        float v = l_run[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        l_run[h] = v;
      }
      float *ls = red + 2 * (4 * DT_N);
      if (!exchange(ls + w4 * DT_N, l_run, lred_full, nq & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      const int d = row;
#pragma unroll
      for (int h = 0; h < RN; ++h) {
        if (h >= a.r) continue;
        const float lsum = ls[h] + ls[DT_N + h] + ls[2 * DT_N + h] + ls[3 * DT_N + h];
        const int hq = g * a.r + h;
        if (a.n_split == 1) {
          a.o[((size_t)b * a.H + hq) * DT_D + d] = __float2bfloat16_rn(ov[h] / lsum);
        } else {
          float *pp = a.part + (((size_t)b * a.H + hq) * a.n_split + k0 / DT_CHUNK) * (DT_D + 2);
          pp[d] = ov[h];
          if (d == 0) {
            pp[DT_D] = m_run[h];
            pp[DT_D + 1] = lsum;
          }
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (a.items != nullptr && threadIdx.x == 0) {
    // every CTA's producer has taken its last item before counting itself done:
    // the last one returns the counters to zero for the next launch
    if (atomicAdd(a.items + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(a.items, 0);
      atomicExch(a.items + 1, 0);
    }
  }
  if (sync.fused()) {  // the next phase reuses this shared memory and TMEM
    if (threadIdx.x == 0) {
      for (int i = 0; i < L::NBAR; ++i) ptx::mbar_inval(b0 + 8u * i);
    }
  } else if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, DtLayout::TMEM_COLS);
  }
}

// Tensor maps and arguments of one decode attention call, exactly as
// launch_attn_decode_tc launches it; n_split > 1 leaves fp32 partials in the
// scratch for the combine step.  For a caller that runs it as a kernel phase.
cudaError_t attn_decode_tc_prepare(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos,
                                   int H, int G, int cache_seq, const AttnScratch &scratch, int *status,
                                   CUtensorMap *mq, CUtensorMap *mk, CUtensorMap *mv, DtArgs *a);

}  // namespace llama
