// Internal launch wrappers of the sm_103a tensor-core (tcgen05 / TMA) kernels
// and the bf16 attention paths.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace llama {

// C[M,N] = epi(A[M,K] W[N,K]^T) on tcgen05 tensor cores, bf16 operands, fp32
// accumulation in TMEM.  Epilogues (kernels.h Epilogue):
//   EPI_STORE    C bf16 [M,N]
//   EPI_RESIDUAL C bf16 [M,N] = R + acc (R bf16 [M,N]; C may equal R)
//   EPI_SWIGLU   W holds gate/up rows interleaved in groups of 16 (see
//                launch_interleave_rows); C bf16 [M, N/2] = SiLU(gate) * up
//   EPI_F32OUT   C fp32 [M,N]
// Requirements: K % 8 == 0 (16-byte TMA row pitch); EPI_SWIGLU needs N % 32 == 0.
// Split-K scratch of the GEMM (fp32 partial tiles and arrival counters).
struct GemmWorkspace {
  float *part = nullptr;
  size_t part_bytes = 0;
  int *counters = nullptr;
  int counter_slots = 0;
};
size_t gemm_splitk_part_bytes();
int gemm_splitk_counter_slots();

// Tile width and K split chosen for a shape (split-K only when ws can hold it):
// few-row shapes split every tile; large shapes split only the tiles of a
// partial last wave.
struct GemmPlan {
  int bn = 256;
  int splits = 1;       // K pieces of each split tile
  int ksteps_split = 0;  // BK steps per piece
  int split_tiles = 0;   // how many tiles (the last ones in raster order) are split
};
// allow_cluster: the GEMM runs as its own launch, which may group a tile's K
// pieces into a thread-block cluster (a phase of a fused kernel cannot).
GemmPlan plan_gemm(int M, int N, int K, size_t ws_part_bytes, int ws_counter_slots, bool allow_cluster = true);

// RMSNorm statistics for the fused epilogues: ss_in (ROWSCALE modes) holds
// sum_j A[m][j]^2 over the d normalised columns; ss_out (EPI_RESIDUAL_SQSUM)
// receives sum_n C[m][n]^2 (must be zero before the launch).
struct RowNorm {
  const float *ss_in = nullptr;
  float *ss_out = nullptr;
  // EPI_RESIDUAL_SQSUM: rows of these arrays (either may be null) are cleared by
  // the epilogue of N tile 0, for accumulators of later kernels whose readers
  // have finished before this kernel starts
  float *zero_a = nullptr, *zero_b = nullptr;
  float eps = 0.f;
  int d = 1;
};

// EPI_QKV_ROPE destinations: GEMM row m is token (b, s) = (m / S, m % S) at
// position p = start_pos + s; output columns [0, H D) are q, [H D, (H+G) D) k
// and [(H+G) D, (H+2G) D) v.  q and k pairs (2i, 2i+1) of each head are
// rotated by table[p][i] = {cos, sin}; rotated q goes to q [T][H D], rotated k
// and v to kc / vc [batch][G][cache_seq][D].  Needs D % 32 == 0.
// halves = 1: the q / k rows of W were reordered by launch_permute_halves_rows,
// so accumulator columns (2i, 2i+1) of a head hold components (i, i + D/2); the
// pair is rotated as above and stored back at i and i + D/2 (natural order).
struct QkvScatter {
  const float2 *table = nullptr;  // launch_rope_table_grouped layout, table_seq positions
  int table_seq = 0;
  bf16 *q = nullptr, *kc = nullptr, *vc = nullptr;
  int S = 1, start_pos = 0, H = 0, G = 0, D = 0, cache_seq = 0, halves = 0;
};

// status: device status word for bounded-wait expiry (may be null).
// ws: split-K scratch (null: never split).  norm: required by the ROWSCALE, SQSUM
// and QKV_ROPE epilogues; scatter: required by EPI_QKV_ROPE (C unused there).
// weights_static: W is not written by any kernel that may still be running
// (library-owned weights), so its first tiles are requested before the kernel
// waits for its predecessor (programmatic dependent launch).
cudaError_t launch_gemm_tc(const bf16 *A, const bf16 *W, const bf16 *R, void *C, int M, int N, int K, int epi,
                           int *status, cudaStream_t st, const GemmWorkspace *ws = nullptr,
                           const RowNorm *norm = nullptr, const QkvScatter *scatter = nullptr,
                           bool weights_static = false);

// Grouped GEMM (one per expert): rows [group_off[g], group_off[g+1]) of A [M][K]
// times rows [g*N, (g+1)*N) of W [n_groups*N][K]; C [M][N] (EPI_STORE) or
// [M][N/2] (EPI_SWIGLU, W rows interleaved per group as for the dense
// gate/up).  group_off (n_groups + 1 ints, device) may be written by the
// preceding kernel on the stream; N must be a multiple of 64.
cudaError_t launch_gemm_grouped(const bf16 *A, const bf16 *W, void *C, int M, int N, int K, int n_groups,
                                const int *group_off, int epi, int *status, cudaStream_t st);

// Reorder the rows of each of `heads` consecutive D-row heads of W [heads*D][d]:
// out row 2i <- row i, out row 2i+1 <- row i + D/2 (the halves RoPE pairs become
// adjacent output columns of x W^T).  d % 8 == 0.
cudaError_t launch_permute_halves_rows(const bf16 *W, bf16 *out, int heads, int D, int d, cudaStream_t st);

// out[32j + i] = gate[16j + i], out[32j + 16 + i] = up[16j + i] (rows of width d), F % 16 == 0.
cudaError_t launch_interleave_rows(const bf16 *gate, const bf16 *up, bf16 *out, int F, int d, cudaStream_t st);

// Scratch of the split-KV decode attention (fp32 partial outputs and row stats).
struct AttnScratch {
  void *partial = nullptr;
  size_t bytes = 0;
  // tensor-core decode attention: two ints, zero between launches (the last CTA
  // of a launch returns them to zero); with them CTAs take work items as they
  // free up instead of a fixed share.  Null: a fixed share per CTA.
  int *item_counters = nullptr;
};
size_t attn_decode_scratch_bytes(int max_tokens, int H, int D, int max_seq);

// Split-KV decode attention (S = 1) -- decode_attn.cu.
bool attn_decode_supported(int H, int G, int D);
cudaError_t launch_attn_decode(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos, int H,
                               int G, int D, int cache_seq, const AttnScratch &scratch, int *status,
                               cudaStream_t st);

// Merge split-KV partials [BH][n_split][D + 2] (o, m, l) into o [BH][D] bf16.
cudaError_t launch_decode_combine(const float *part, bf16 *o, int BH, int D, int n_split, cudaStream_t st);

// Tensor-core decode attention (D = 128) -- decode_tc.cu.
bool attn_decode_tc_supported(int H, int G, int D);
size_t attn_decode_tc_scratch_bytes(int B, int H, int kv_len);
cudaError_t launch_attn_decode_tc(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int start_pos,
                                  int H, int G, int cache_seq, const AttnScratch &scratch, int *status,
                                  cudaStream_t st);

// The decode step (S = 1) of a dense bf16 block with d_head = 128 as one
// cooperative kernel (decode_fused.cu): attention-norm statistics, QKV GEMM +
// RoPE + cache write, decode attention, chunk merge, O GEMM + residual, gate/up
// GEMM + SwiGLU, down GEMM + residual, separated by grid-wide barriers.  The
// buffers and weights are those of the multi-kernel path (weights as repacked
// at create: norm gains folded, gate/up interleaved).  sync: two device words
// of this handle (cleared by the launch).
struct DecodeFusedParams {
  const bf16 *x = nullptr;  // [B][d]
  bf16 *y = nullptr;        // [B][d]
  const bf16 *wqkv = nullptr, *wo = nullptr, *w_gu = nullptr, *w_down = nullptr;
  bf16 *q = nullptr, *o = nullptr, *h = nullptr, *act = nullptr;  // workspace activations
  float *ss_x = nullptr, *ss_h = nullptr;
  const float2 *rope = nullptr;  // launch_rope_table_grouped layout, rope_seq positions
  int rope_seq = 0;
  bf16 *kc = nullptr, *vc = nullptr;
  int cache_seq = 0;
  int B = 0, start_pos = 0, d = 0, H = 0, G = 0, D = 0, F = 0, halves = 0;
  float eps = 0.f;
  GemmWorkspace gemm;
  AttnScratch attn;
  unsigned *sync = nullptr;
  int *status = nullptr;
};
// True when this device can run the fused kernel (cooperative launch with one
// CTA per SM).
bool decode_fused_available();
cudaError_t launch_decode_block_fused(const DecodeFusedParams &p, cudaStream_t st);

// Causal GQA attention over the bf16 cache; picks the prefill or decode kernel.
cudaError_t launch_attention(const bf16 *q, const bf16 *kc, const bf16 *vc, bf16 *o, int B, int S, int start_pos,
                             int H, int G, int D, int cache_seq, const AttnScratch &scratch, int *status,
                             cudaStream_t st);

}  // namespace llama
