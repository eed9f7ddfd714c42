// Causal grouped-query attention over the bf16 KV cache on tcgen05 tensor cores
// ("The Evolving Transformer 04 · LLaMA", §05 GQA; "Full Llama 3 transformer
// block", How it works: cache read with the start_pos offset mask).
//
// Prefill kernel (persistent, at most one CTA per SM, 320 threads; each CTA
// loops over work items (sequence b, KV head g, block of 2*Mq query positions)
// and the next item's Q, first K tile and first S products overlap the current
// item's last PV products and output):
//   * A 128-row query tile packs the r = H/G query heads of group g: row
//     hh*Mq + i is head g*r + hh at position q0 + i (Mq = 128 / r rounded down
//     to a multiple of 8; rows past r*Mq are zero).  Each K/V tile that lands in shared memory therefore
//     serves every query head of its group; the CTA holds two such tiles
//     (t = 0, 1: consecutive position blocks) that ping-pong.
//   * warp 0: TMA producer -- Q tiles once, then 128-key K and V tiles into a
//     two-stage ring.  K/V tensor maps end at start_pos + S, so keys beyond
//     the valid cache read as zeros.
//   * warp 1: tcgen05.mma issuer -- S_t = Q_t K^T (fp32 in TMEM), then
//     O_t += P_t V with P_t read from TMEM and V as an MN-major smem operand.
//   * warps 2-5 / 6-9: softmax of tile 0 / 1, one thread per row, one pass
//     over each S row in TMEM: causal mask j <= start_pos + position, running
//     max (rescaling only when it grows by more than 2^8; the max of each
//     32-column chunk comes from the TMEM load's own reduction),
//     p = 2^(s*log2e/sqrt(D) - m) on the MUFU unit, P written back to TMEM as
//     bf16 over its own S columns; finally O / l stored as bf16.
// Every wait is bounded; on expiry the kernel records a status code, drains,
// frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tc_kernels.h"

namespace llama {
namespace {

constexpr int ATT_THREADS = 320;
constexpr int KV_TILE = 128;
constexpr int KV_STAGES = 2;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units: rescale O when the running max grows by > 2^8
// Of every 32 exponentials of a row, this many run as a polynomial on the FMA
// pipe and the rest on the MUFU unit.  Measured on GB300 at the 8B prefill
// shape: 0 of 32 is fastest (the MUFU unit is not what paces the tile), so the
// polynomial path is off by default; -DLLAMA_POLY_EXP2_PER_32=n turns it on.
#ifndef LLAMA_POLY_EXP2_PER_32
#define LLAMA_POLY_EXP2_PER_32 0
#endif
constexpr int POLY_EXP2_PER_32 = LLAMA_POLY_EXP2_PER_32;

template <int D>
struct AttnLayout {
  static constexpr int ATOM = 128 * 128;         // one 64-column (128-byte) swizzle atom of 128 rows
  static constexpr int Q_TILE = (D / 64) * ATOM;  // 128 rows x D
  static constexpr int KV_BYTES = (D / 64) * ATOM;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * Q_TILE;
  static constexpr int OFF_V = OFF_K + KV_STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + KV_STAGES * KV_BYTES;
  // q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], o_done[2], fin, q_empty
  static constexpr int NBAR = 1 + 4 * KV_STAGES + 6 + 1 + 1;
  // At least 116 KB so that a second CTA never shares the SM (both would need all 512 TMEM columns).
  static constexpr int BYTES_MIN = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int BYTES = BYTES_MIN > 116 * 1024 ? BYTES_MIN : 116 * 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S0, S1 (128 each), O0, O1 (D each)
};

struct AttnArgs {
  bf16 *o;
  int B, S, start_pos, H, G, r, Mq, kv_len, nqb;
  float scale_log2;
  int *status;
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, AttnArgs a) {
  using L = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t s0 = ptx::smem_u32(smem);
  const uint32_t bar0 = ptx::smem_u32(bars);
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + KV_STAGES + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * KV_STAGES + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * KV_STAGES + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (1 + 4 * KV_STAGES + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (3 + 4 * KV_STAGES + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (5 + 4 * KV_STAGES + t); };
  const uint32_t fin = bar0 + 8u * (7 + 4 * KV_STAGES);
  const uint32_t q_empty = bar0 + 8u * (8 + 4 * KV_STAGES);  // the MMAs reading an item's Q are done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Persistent CTAs: the CTA takes the items (b, g, block of 2*Mq positions)
  // blockIdx.x, then one per round in snake order over the grid (rounds
  // alternate direction), longest query blocks first, so that the CTAs' sums of
  // key tiles even out.  Barrier phases run on across items: a role's counters
  // (items started, key tiles issued) give every wait its parity.
  const int bg_count = a.B * a.G;
  const int n_items = a.nqb * bg_count;
  auto item_of = [&](int k) -> int {  // the CTA's k-th item, -1 past the last
    const int gsz = (int)gridDim.x;
    const int u = k * gsz + ((k & 1) ? gsz - 1 - (int)blockIdx.x : (int)blockIdx.x);
    return u < n_items ? u : -1;
  };
  struct Item {
    int b, g, q0, n_kv;
  };
  auto decode_item = [&](int u) {
    Item it;
    const int qb = a.nqb - 1 - u / bg_count;
    const int bg = u % bg_count;
    it.b = bg / a.G;
    it.g = bg % a.G;
    it.q0 = qb * 2 * a.Mq;
    const int kv_need = min(a.start_pos + it.q0 + 2 * a.Mq, a.kv_len);
    it.n_kv = (kv_need + KV_TILE - 1) / KV_TILE;
    return it;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int s = 0; s < KV_STAGES; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
      ptx::mbar_init(v_full(s), 1);
      ptx::mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(s_full(t), 1);
      ptx::mbar_init(p_full(t), 128);
      ptx::mbar_init(o_done(t), 1);
    }
    ptx::mbar_init(fin, 1);
    ptx::mbar_init(q_empty, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  // Query-head slots beyond r (r not a power of two) are never loaded: zero them.
  if (warp >= 2 && a.r * a.Mq < 128) {
    const int first = a.r * a.Mq;
    for (int t = 0; t < 2; ++t)
      for (int at = 0; at < D / 64; ++at) {
        uint4 *p = reinterpret_cast<uint4 *>(smem + L::OFF_Q + t * L::Q_TILE + at * L::ATOM + first * 128);
        const int n16 = (128 - first) * 8;
        for (int i = threadIdx.x - 64; i < n16; i += ATT_THREADS - 64) p[i] = make_uint4(0, 0, 0, 0);
      }
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // programmatic dependent launch: q and the cache come from earlier kernels
  allow_dependents_launch();
  grid_dependency_wait();

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      const uint32_t qbytes = 2u * a.r * (D / 64) * a.Mq * 128u;
      int items = 0;   // Q loads issued
      int issued = 0;  // K and V loads issued over all items: 2 per key tile
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = item_of(k);
        if (u < 0) break;
        const Item it = decode_item(u);
        // the previous item's Q stays until its last S product is done
        if (k > 0 && !ptx::mbar_wait(q_empty, (k - 1) & 1, abort_flag, a.status, DEV_TIMEOUT_PRODUCER)) break;
        ptx::mbar_arrive_expect_tx(q_full, qbytes);
        for (int t = 0; t < 2; ++t)
          for (int hh = 0; hh < a.r; ++hh)
            for (int at = 0; at < D / 64; ++at)
              ptx::tma_load_4d(s0 + L::OFF_Q + t * L::Q_TILE + at * L::ATOM + hh * a.Mq * 128, &tmQ, at * 64,
                               it.g * a.r + hh, it.q0 + t * a.Mq, it.b, q_full);
        ++items;
        for (int j = 0; j < it.n_kv; ++j) {
          const int jj = issued / 2;  // key tile index over all items
          const int st = jj % KV_STAGES;
          const uint32_t ph = (jj / KV_STAGES) & 1;
          if (!ptx::mbar_wait(k_empty(st), ph ^ 1, abort_flag, a.status, DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(k_full(st), L::KV_BYTES);
          for (int at = 0; at < D / 64; ++at)
            ptx::tma_load_4d(s0 + L::OFF_K + st * L::KV_BYTES + at * L::ATOM, &tmK, at * 64, j * KV_TILE, it.g,
                             it.b, k_full(st));
          ++issued;
          if (!ptx::mbar_wait(v_empty(st), ph ^ 1, abort_flag, a.status, DEV_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(v_full(st), L::KV_BYTES);
          for (int at = 0; at < D / 64; ++at)
            ptx::tma_load_4d(s0 + L::OFF_V + st * L::KV_BYTES + at * L::ATOM, &tmV, at * 64, j * KV_TILE, it.g,
                             it.b, v_full(st));
          ++issued;
        }
      }
      // Drain: every issued copy must land before the CTA exits (at most one Q
      // load and the ring's last KV_STAGES key tiles can be outstanding).
      if (items > 0) ptx::mbar_drain(q_full, (items - 1) & 1, a.status, DEV_TIMEOUT_PRODUCER);
      for (int j = max(0, issued / 2 - KV_STAGES); j < (issued + 1) / 2; ++j) {
        const int st = j % KV_STAGES;
        const uint32_t ph = (j / KV_STAGES) & 1;
        ptx::mbar_drain(k_full(st), ph, a.status, DEV_TIMEOUT_PRODUCER);
        if (2 * j + 1 < issued) ptx::mbar_drain(v_full(st), ph, a.status, DEV_TIMEOUT_PRODUCER);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, KV_TILE, false);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, true);
      // S_t(j) = Q_t K(j)^T into TMEM columns t*128 (P_t later overwrites them as bf16);
      // j counts key tiles over all items (it picks the ring stage).
      auto issue_s = [&](int j, int t) {
        const uint32_t kb = s0 + L::OFF_K + (j % KV_STAGES) * L::KV_BYTES;
        const uint32_t qbase = s0 + L::OFF_Q + t * L::Q_TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * L::ATOM + (kk % 4) * 32;
          ptx::mma_bf16_ss(tmem + t * 128, ptx::smem_desc_sw128(qbase + off), ptx::smem_desc_sw128(kb + off),
                           idesc_qk, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full(t));
      };
      // O_t += P_t(j) V(j), P_t read from TMEM, V as an MN-major operand; the item's
      // first key tile (first = true) overwrites O.
      auto issue_pv = [&](int j, bool first, int t) {
        const uint32_t vb = s0 + L::OFF_V + (j % KV_STAGES) * L::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < KV_TILE / 16; ++kk) {
          // 16 keys = two 8-row groups of the V tile; V rows hold 64 consecutive d values.
          const uint64_t bdesc = ptx::smem_desc_sw128_mn(vb + kk * 16 * 128, L::ATOM, 1024);
          ptx::mma_bf16_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8, bdesc, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(o_done(t));
      };
      // Staggered order: S_0(j+1) is issued right after PV_0(j), so the softmax of tile 0 for
      // the next key tile overlaps the softmax of tile 1 and the tensor core alternates tiles.
      // The next item's first S products follow the last PV products of the current one
      // (MMAs of one thread run in issue order), so they overlap the current item's epilogue.
      // q_empty is committed after an item's last S products.
      bool ok = true;
      int jg = 0;  // key tiles consumed over all items
      for (int k = 0; ok; ++k) {
        const int u = item_of(k);
        if (u < 0) break;
        const int n_kv = decode_item(u).n_kv;
        if (!ptx::mbar_wait(q_full, k & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
        if (!ptx::mbar_wait(k_full(jg % KV_STAGES), (jg / KV_STAGES) & 1, abort_flag, a.status, DEV_TIMEOUT_MMA))
          break;
        ptx::tc_fence_after();
        issue_s(jg, 0);
        issue_s(jg, 1);
        ptx::mma_commit(k_empty(jg % KV_STAGES));
        if (n_kv == 1) ptx::mma_commit(q_empty);
        for (int j = 0; j < n_kv; ++j) {
          const int jj = jg + j;
          const int st = jj % KV_STAGES;
          const uint32_t ph = (jj / KV_STAGES) & 1;
          ok = false;
          if (!ptx::mbar_wait(v_full(st), ph, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
          if (!ptx::mbar_wait(p_full(0), jj & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
          ptx::tc_fence_after();
          issue_pv(jj, j == 0, 0);
          const bool more = j + 1 < n_kv;
          if (more) {
            const int st1 = (jj + 1) % KV_STAGES;
            if (!ptx::mbar_wait(k_full(st1), ((jj + 1) / KV_STAGES) & 1, abort_flag, a.status, DEV_TIMEOUT_MMA))
              break;
            ptx::tc_fence_after();
            issue_s(jj + 1, 0);
          }
          if (!ptx::mbar_wait(p_full(1), jj & 1, abort_flag, a.status, DEV_TIMEOUT_MMA)) break;
          ptx::tc_fence_after();
          issue_pv(jj, j == 0, 1);
          ptx::mma_commit(v_empty(st));
          if (more) {
            issue_s(jj + 1, 1);
            ptx::mma_commit(k_empty((jj + 1) % KV_STAGES));
            if (j + 2 == n_kv) ptx::mma_commit(q_empty);
          }
          ok = true;
        }
        jg += n_kv;
      }
      ptx::mma_commit(fin);
      ptx::mbar_drain(fin, 0, a.status, DEV_TIMEOUT_MMA);
    }
  } else {
    // ---------------------------------------------------------- softmax ---
    const int t = (warp - 2) / 4;
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int hh = row / a.Mq, i = row % a.Mq;
    const uint32_t lane_base = tmem + ((uint32_t)(qq * 32) << 16);
    const uint32_t s_col = lane_base + t * 128;
    const uint32_t o_col = lane_base + 256 + t * D;
    const uint64_t scale2 = ptx::f2pack(a.scale_log2, a.scale_log2);
    bool ok = true;
    int jg = 0;  // key tiles of earlier items (the phase count of s_full, p_full and o_done)
    for (int k = 0; ok; ++k) {
      const int u = item_of(k);
      if (u < 0) break;
      const Item it = decode_item(u);
      const int n_kv = it.n_kv;
      const int rel = it.q0 + t * a.Mq + i;
      const bool valid = hh < a.r && rel < a.S;
      const int pos = a.start_pos + rel;
      float m_run = -INFINITY;
      uint64_t l2 = ptx::f2pack(0.f, 0.f);  // running row sum, two partial halves
      for (int j = 0; j < n_kv; ++j) {
        ok = ptx::mbar_wait(s_full(t), (jg + j) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // One pass over the tile, 32 columns at a time.  p = 2^(s*scale - m_run)
        // uses the running maximum as it stands; a chunk whose own maximum exceeds
        // it by more than 2^8 first raises it (the rescale), scaling the row sum,
        // the P chunks already written for this tile and, once the tile is done,
        // O.  The chunk maximum comes from the TMEM load itself; the causal
        // predicate applies only on tiles that reach past some row's position.
        // The P chunk of columns [c, c+32) lands in TMEM columns [c/2, c/2 + 16),
        // which hold S values already read (columns < c + 32).
        const int key0 = j * KV_TILE;
        const bool masked = __any_sync(0xffffffffu, key0 + KV_TILE - 1 > pos);
        float alpha_tile = 1.f;
        bool rescaled = false;  // warp-uniform
  #pragma unroll
        for (int c = 0; c < KV_TILE; c += 32) {
          float sv[32];
          float cm;
          if (masked) {
            ptx::tmem_ld32(s_col + c, sv);
            cm = -INFINITY;
  #pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (key0 + c + k > pos) sv[k] = -INFINITY;
              cm = fmaxf(cm, sv[k]);
            }
          } else {
            ptx::tmem_ld32_max(s_col + c, sv, cm);
          }
          const float cms = cm * a.scale_log2;
          const bool need = cms > m_run + RESCALE_THRESHOLD;
          if (__any_sync(0xffffffffu, need)) {
            float alpha = 1.f;
            if (need) {
              alpha = ptx::ex2_approx(m_run - cms);
              m_run = cms;
            }
            l2 = ptx::fmul2(l2, ptx::f2pack(alpha, alpha));
            alpha_tile *= alpha;
            rescaled = true;
            if (c > 0) {
              // this tile's P columns written so far were scaled by the old maximum
              ptx::tmem_st_wait();
  #pragma unroll 1
              for (int pc = 0; pc < c / 2; pc += 16) {
                float pv[16];
                ptx::tmem_ld16(s_col + pc, pv);
                uint32_t w[16];
  #pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const uint32_t u = __float_as_uint(pv[e]);
                  w[e] = pack2(__uint_as_float(u << 16) * alpha, __uint_as_float(u & 0xffff0000u) * alpha);
                }
                ptx::tmem_st16(s_col + pc, w);
              }
            }
          }
          const uint64_t negm2 = ptx::f2pack(-m_run, -m_run);
          uint32_t pk[16];
          uint64_t lc = ptx::f2pack(0.f, 0.f);  // this chunk's sum: a second, independent add chain
  #pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float x0, x1, p0, p1;
            ptx::f2unpack(ptx::ffma2(ptx::f2pack(sv[k], sv[k + 1]), scale2, negm2), x0, x1);
            if (k < POLY_EXP2_PER_32) {
              ptx::exp2_poly2(x0, x1, p0, p1);  // FMA pipe
            } else {
              p0 = ptx::ex2_approx(x0);         // MUFU
              p1 = ptx::ex2_approx(x1);
            }
            if ((k & 2) == 0)
              l2 = ptx::fadd2(l2, ptx::f2pack(p0, p1));
            else
              lc = ptx::fadd2(lc, ptx::f2pack(p0, p1));
            pk[k / 2] = pack2(p0, p1);
          }
          l2 = ptx::fadd2(l2, lc);
          ptx::tmem_st16(s_col + c / 2, pk);
        }
        if (j > 0 && rescaled) {
          // O holds the sum over earlier key tiles: wait for the last PV product
          // into it, then scale it by this tile's factor
          ok = ptx::mbar_wait(o_done(t), (jg + j - 1) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
  #pragma unroll
          for (int c = 0; c < D; c += 16) {
            float ov[16];
            ptx::tmem_ld16(o_col + c, ov);
            uint32_t w[16];
  #pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(ov[e] * alpha_tile);
            ptx::tmem_st16(o_col + c, w);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full(t));
      }
      if (ok && n_kv > 0) {
        ok = ptx::mbar_wait(o_done(t), (jg + n_kv - 1) & 1, abort_flag, a.status, DEV_TIMEOUT_ATTN);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          ptx::tc_fence_after();
          float la, lb;
          ptx::f2unpack(l2, la, lb);
          const float inv = 1.f / (la + lb);
          bf16 *dst = a.o + (((size_t)it.b * a.S + rel) * a.H + it.g * a.r + hh) * D;
  #pragma unroll
          for (int c = 0; c < D; c += 16) {
            float ov[16];
            ptx::tmem_ld16(o_col + c, ov);
            ptx::tmem_ld_wait();
            if (valid) {
              uint4 w0 = make_uint4(pack2(ov[0] * inv, ov[1] * inv), pack2(ov[2] * inv, ov[3] * inv),
                                    pack2(ov[4] * inv, ov[5] * inv), pack2(ov[6] * inv, ov[7] * inv));
              uint4 w1 = make_uint4(pack2(ov[8] * inv, ov[9] * inv), pack2(ov[10] * inv, ov[11] * inv),
                                    pack2(ov[12] * inv, ov[13] * inv), pack2(ov[14] * inv, ov[15] * inv));
              *reinterpret_cast<uint4 *>(dst + c) = w0;
              *reinterpret_cast<uint4 *>(dst + c + 8) = w1;
            }
          }
        }
      }
      jg += n_kv;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
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

// 4-D bf16 map, dims/strides innermost first (strides in bytes for dims 1..3), box {64, b1, b2, 1}.
bool make_map_4d(CUtensorMap *map, const void *ptr, const uint64_t dims[4], const uint64_t strides[3], uint32_t b1,
                 uint32_t b2) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gstride[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t box[4] = {64, b1, b2, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prefill(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int S, int start_pos,
                           int H, int G, int cache_seq, int *status, cudaStream_t st) {
  using L = AttnLayout<D>;
  static PerContextOnce attr;
  const cudaError_t attr_err = attr.run([] {
    return cudaFuncSetAttribute(attn_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int r = H / G;
  // positions per query tile: as many as the r heads fill of its 128 rows, a
  // multiple of 8 so that every head's Q box starts on a 1024-byte swizzle atom
  // (r = 3: 40 positions, 120 rows; r = 5: 24 positions, 120 rows)
  const int Mq = (128 / r) & ~7;
  const int kv_len = start_pos + S;
  CUtensorMap mq, mk, mv;
  const uint64_t qd[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)S, (uint64_t)B};
  const uint64_t qs[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)S * H * D * 2};
  const uint64_t kd[4] = {(uint64_t)D, (uint64_t)kv_len, (uint64_t)G, (uint64_t)B};
  const uint64_t ks[3] = {(uint64_t)D * 2, (uint64_t)cache_seq * D * 2, (uint64_t)G * cache_seq * D * 2};
  if (!make_map_4d(&mq, q, qd, qs, 1, Mq) || !make_map_4d(&mk, kc, kd, ks, KV_TILE, 1) ||
      !make_map_4d(&mv, vc, kd, ks, KV_TILE, 1))
    return cudaErrorInvalidValue;
  AttnArgs args;
  args.o = o;
  args.B = B;
  args.S = S;
  args.start_pos = start_pos;
  args.H = H;
  args.G = G;
  args.r = r;
  args.Mq = Mq;
  args.kv_len = kv_len;
  args.nqb = (S + 2 * Mq - 1) / (2 * Mq);
  args.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  args.status = status;
  // persistent: at most one CTA per SM, each looping over its items
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int items = B * G * args.nqb;
  const unsigned grid = (unsigned)(sms > 0 && sms < items ? sms : items);
  count_launch();
  return launch_pdl(attn_prefill_kernel<D>, dim3(grid), dim3(ATT_THREADS), L::BYTES, st, mq, mk, mv, args);
}

}  // namespace

cudaError_t launch_attention(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int S, int start_pos,
                             int H, int G, int D, int cache_seq, const AttnScratch &scratch, int *status,
                             cudaStream_t st) {
  const int r = H / G;
  if (S == 1 && attn_decode_tc_supported(H, G, D) &&
      (start_pos + 1 <= 512 || scratch.bytes >= attn_decode_tc_scratch_bytes(B, H, start_pos + 1)))
    return launch_attn_decode_tc(q, kc, vc, o, B, start_pos, H, G, cache_seq, scratch, status, st);
  if (S == 1 && attn_decode_supported(H, G, D))
    return launch_attn_decode(q, kc, vc, o, B, start_pos, H, G, D, cache_seq, scratch, status, st);
  const bool tc_ok = (D == 64 || D == 128) && r <= 8 && S > 1;
  if (tc_ok) {
    if (D == 128) return launch_prefill<128>(q, kc, vc, o, B, S, start_pos, H, G, cache_seq, status, st);
    return launch_prefill<64>(q, kc, vc, o, B, S, start_pos, H, G, cache_seq, status, st);
  }
  return launch_attention_simt<bf16>(q, kc, vc, o, B, S, start_pos, H, G, D, cache_seq, st);
}

}  // namespace llama
