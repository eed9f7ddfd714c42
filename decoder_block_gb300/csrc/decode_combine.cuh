// Merge of split-KV decode attention partials, shared by the combine kernel
// (decode_attn.cu) and the fused decode-step kernel (decode_fused.cu).
// "Full Llama 3 transformer block", How it works: each query attends to every
// cached key; the keys are processed in chunks whose softmax partials
// (o = sum_j 2^(s_j - m) v_j, m, l = sum_j 2^(s_j - m)) combine exactly:
//   o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c,   M = max_c m_c.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace llama {

// Output element d of (b, h) row bh: part [BH][n_split][D + 2] (o[D], m, l).
template <int D>
__device__ __forceinline__ void decode_combine_element(const float *__restrict__ part, bf16 *__restrict__ o, int bh,
                                                       int d, int n_split) {
  const float *p = part + (size_t)bh * n_split * (D + 2);
  float m = -INFINITY;
  for (int s = 0; s < n_split; ++s) m = fmaxf(m, p[s * (D + 2) + D]);
  float ov = 0.f, lv = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float ms = p[s * (D + 2) + D];
    const float f = (ms == -INFINITY) ? 0.f : ptx::ex2_approx(ms - m);
    ov = fmaf(f, p[s * (D + 2) + d], ov);
    lv = fmaf(f, p[s * (D + 2) + D + 1], lv);
  }
  o[(size_t)bh * D + d] = __float2bfloat16_rn(ov / lv);
}

}  // namespace llama
