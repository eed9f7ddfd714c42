// Host runtime behind the C ABI: argument validation, weight repacking,
// workspace ownership and the per-forward kernel sequence.
//
// Forward sequence of one block ("Full Llama 3 transformer block", How it
// works; "The Evolving Transformer 04 · LLaMA", §06 Block):
//   1. u   = RMSNorm(x; attention_norm)
//   2. qkv = u [Wq; Wk; Wv]^T                 (one fused projection)
//   3. q   = RoPE(q); K cache <- RoPE(k); V cache <- v   at start_pos + s
//   4. o   = causal GQA attention over the cache
//   5. h   = x + o Wo^T                       (residual in the epilogue)
//   6. v2  = RMSNorm(h; ffn_norm)
//   7. a   = SiLU(v2 W_gate^T) * (v2 W_up^T)  (SwiGLU in the epilogue)
//   8. y   = h + a W_down^T                   (residual in the epilogue)
// bf16 tensor-core path: both RMSNorms are fused -- their gains are folded into
// [Wq; Wk; Wv] and [W_gate; W_up] at create time, a row-statistics pass (step 1)
// and the O-projection epilogue (step 5) produce sum(x^2) and sum(h^2) per row,
// and the QKV and gate/up epilogues scale each row by rsqrt(mean + eps).  The
// QKV epilogue also applies RoPE and writes k and v into the cache (step 3 in
// the same kernel as step 2, for d_head % 32 == 0).  The fp32 path keeps the
// standalone steps.
#include <cuda.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "llama_block.h"
#include "kernels.h"
#include "tc_kernels.h"

using namespace llama;

namespace {
thread_local const char *t_last_cuda_error = "no error";
}  // namespace

namespace llama {
void note_cuda_error(cudaError_t e) { t_last_cuda_error = cudaGetErrorString(e); }

std::atomic<unsigned long long> g_kernel_launches{0};
void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned long long current_context_id() {
  typedef CUresult (*GetCurrent)(CUcontext *);
  typedef CUresult (*GetId)(CUcontext, unsigned long long *);
  static const std::pair<GetCurrent, GetId> fns = []() {
    void *cur = nullptr, *id = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess)
      cur = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      id = nullptr;
    cudaGetLastError();
    return std::make_pair(reinterpret_cast<GetCurrent>(cur), reinterpret_cast<GetId>(id));
  }();
  if (fns.first == nullptr || fns.second == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr || fns.second(ctx, &v) != CUDA_SUCCESS) return 0;
  return v;
}
}  // namespace llama

namespace {

struct Dims {
  int d, H, G, D, F, QKV, max_seq;
  float eps;
  double theta;
  RopeScaling rope_scaling;
  int rope_halves;          // pairs (i, i + D/2) instead of (2i, 2i+1)
  int E = 0, topk = 0, Fs = 0, E_pad = 0;  // mixture of experts (E = 0: dense); router rows padded to 64
  int dtype;
  size_t esize;
  bool moe() const { return E > 0; }
  // halves RoPE on the fused QKV epilogue: the q / k rows of Wqkv are stored
  // reordered so that each pair lands in adjacent accumulator columns
  bool fused_qkv_rope() const { return dtype == LLAMA_BF16 && D % 32 == 0; }
  bool permute_halves() const { return rope_halves && fused_qkv_rope(); }
};

// Device allocations owned by one handle, freed together.
struct Allocs {
  std::vector<void *> ptrs;
  bool failed = false;
  void *alloc(size_t bytes) {
    void *p = nullptr;
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      failed = true;
      cudaGetLastError();
      return nullptr;
    }
    ptrs.push_back(p);
    return p;
  }
  void free_all() {
    for (void *p : ptrs) cudaFree(p);
    ptrs.clear();
  }
};

struct Weights {
  void *attn_norm = nullptr, *ffn_norm = nullptr;
  void *wqkv = nullptr;  // [(H + 2G) D, d]: rows of Wq, then Wk, then Wv
  void *wo = nullptr;    // [d, H D]
  void *w_gate = nullptr, *w_up = nullptr;  // [F, d] each
  void *w_gu = nullptr;  // bf16 tensor-core path: gate/up rows interleaved per 16-row group, [2F, d]
  void *w_down = nullptr;  // [d, F]  (mixture of experts: [E d, F], one [d, F] slice per expert)
  // mixture of experts: w_gu holds every expert's interleaved gate/up rows [E 2F, d];
  // router [E_pad, d] with the ffn-norm gain folded in (rows >= E zero);
  // shared expert: gate/up interleaved with the gain folded in [2 Fs, d], down [d, Fs]
  void *router = nullptr, *shared_gu = nullptr, *shared_down = nullptr;
};

struct Workspace {
  int max_tokens = 0;
  void *xn = nullptr, *qkv = nullptr, *q = nullptr, *o = nullptr, *h = nullptr, *act = nullptr, *hn = nullptr;
  void *xin = nullptr, *yout = nullptr;  // staging for the host-buffer entry point
  AttnScratch attn;                      // split-KV partials of the decode path
  GemmWorkspace gemm;                    // split-K partials of few-row GEMMs (decode)
  float *ss_x = nullptr, *ss_h = nullptr;  // per-row sums of squares (fused RMSNorm statistics)
  float *ss_x2 = nullptr;                  // the other input-statistics buffer of a stack's layer chain
  // mixture of experts: router logits [T][E_pad] fp32; per (token, choice) expert id,
  // weight and row in the expert-grouped buffers; per-expert counts / offsets / fill;
  // expert inputs [T k][d], SwiGLU outputs [T k][F], outputs [T k][d]; shared expert
  // activations [T][Fs] and h + shared [T][d]
  float *logits = nullptr, *route_w = nullptr;
  int *route_ids = nullptr, *route_pos = nullptr, *counts = nullptr, *offsets = nullptr, *fill = nullptr;
  void *xin_e = nullptr, *act_e = nullptr, *y_e = nullptr, *act_s = nullptr, *hs = nullptr;
  int last_tokens = 0;  // B * S of the most recent forward (routing introspection)
  unsigned *fused_sync = nullptr;  // phase barrier words of the fused decode kernel
  int decode_mode = LLAMA_DECODE_KERNELS;
};

// Optional per-step event timing of block forwards (llama_block_profile_*).
struct Profiler {
  bool on = false;
  int max_forwards = 0, used = 0;
  std::vector<cudaEvent_t> ev;  // [max_forwards][LLAMA_PROFILE_STEPS][2]
  std::vector<char> launched;   // [max_forwards][LLAMA_PROFILE_STEPS]: the step launched a kernel
  cudaEvent_t *slot = nullptr;  // events of the forward being enqueued (null: not recording)
  char *slot_launched = nullptr;
  unsigned long long at_begin = 0;  // library launch count at the step's first edge
  void begin_forward() {
    slot = (on && used < max_forwards) ? &ev[(size_t)used * LLAMA_PROFILE_STEPS * 2] : nullptr;
    slot_launched = slot != nullptr ? &launched[(size_t)used * LLAMA_PROFILE_STEPS] : nullptr;
    if (slot != nullptr) ++used;
  }
  // A step fused into another step's kernel launches nothing between its two
  // edges; it is then left out of the per-step times.
  void mark(int step, int edge, cudaStream_t st) {
    if (slot == nullptr) return;
    cudaEventRecord(slot[step * 2 + edge], st);
    const unsigned long long n = g_kernel_launches.load(std::memory_order_relaxed);
    if (edge == 0)
      at_begin = n;
    else
      slot_launched[step] = n != at_begin ? 1 : 0;
  }
  void release() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    launched.clear();
    on = false;
    used = max_forwards = 0;
    slot = nullptr;
    slot_launched = nullptr;
  }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_device_ptr(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

llama_status check_ptr(const void *p) {
  if (p == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(p)) return LLAMA_ERR_ALIGN;
  if (!is_device_ptr(p)) return LLAMA_ERR_INVALID_ARG;
  return LLAMA_OK;
}

llama_status validate_config(const llama_config *c, Dims *dm) {
  if (c == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (c->dtype != LLAMA_F32 && c->dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->d_ff <= 0 || c->max_seq_len <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (!(c->norm_eps >= 0.f) || !(c->rope_theta > 0.f)) return LLAMA_ERR_INVALID_ARG;
  if (c->d_model % c->n_heads != 0) return LLAMA_ERR_SHAPE;
  if (c->n_heads % c->n_kv_heads != 0) return LLAMA_ERR_SHAPE;
  const int D = c->d_model / c->n_heads;
  if (D % 2 != 0) return LLAMA_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return LLAMA_ERR_UNSUPPORTED;
  if (c->rope_layout != LLAMA_ROPE_INTERLEAVED && c->rope_layout != LLAMA_ROPE_HALVES) return LLAMA_ERR_INVALID_ARG;
  const bool scaled = c->rope_scaling_factor > 1.f;
  if (!scaled && !(c->rope_scaling_factor <= 1.f)) return LLAMA_ERR_INVALID_ARG;  // NaN
  if (scaled && !(c->rope_low_freq_factor > 0.f && c->rope_high_freq_factor > c->rope_low_freq_factor &&
                  c->rope_original_max_pos > 0))
    return LLAMA_ERR_INVALID_ARG;
  const int vec = c->dtype == LLAMA_BF16 ? 8 : 4;
  if (c->d_model % vec != 0 || c->d_ff % vec != 0) return LLAMA_ERR_UNSUPPORTED;
  if (c->rope_layout == LLAMA_ROPE_HALVES && (D / 2) % vec != 0) return LLAMA_ERR_UNSUPPORTED;
  if (c->n_experts < 0 || c->top_k < 0 || c->d_ff_shared < 0) return LLAMA_ERR_INVALID_ARG;
  if (c->n_experts > 0) {
    if (c->top_k < 1 || !moe_supported(c->n_experts, c->top_k)) return LLAMA_ERR_INVALID_ARG;
    if (c->dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
    if (c->d_model % 64 != 0 || c->d_ff % 32 != 0 || c->d_ff_shared % 32 != 0) return LLAMA_ERR_UNSUPPORTED;
  }
  if (c->dtype == LLAMA_BF16 && c->d_ff % 16 != 0) return LLAMA_ERR_UNSUPPORTED;  // gate/up interleave groups
  dm->d = c->d_model;
  dm->H = c->n_heads;
  dm->G = c->n_kv_heads;
  dm->D = D;
  dm->F = c->d_ff;
  dm->QKV = (c->n_heads + 2 * c->n_kv_heads) * D;
  dm->max_seq = c->max_seq_len;
  dm->eps = c->norm_eps;
  dm->theta = (double)c->rope_theta;
  dm->rope_halves = c->rope_layout == LLAMA_ROPE_HALVES ? 1 : 0;
  dm->rope_scaling = RopeScaling();
  if (scaled) {
    dm->rope_scaling.factor = (double)c->rope_scaling_factor;
    dm->rope_scaling.low = (double)c->rope_low_freq_factor;
    dm->rope_scaling.high = (double)c->rope_high_freq_factor;
    dm->rope_scaling.original_max_pos = (double)c->rope_original_max_pos;
  }
  dm->E = c->n_experts;
  dm->topk = c->n_experts > 0 ? c->top_k : 0;
  dm->Fs = c->n_experts > 0 ? c->d_ff_shared : 0;
  dm->E_pad = (dm->E + 63) / 64 * 64;
  dm->dtype = c->dtype;
  dm->esize = c->dtype == LLAMA_BF16 ? 2 : 4;
  return LLAMA_OK;
}

llama_status copy_weights(const Dims &dm, const llama_block_weights *w, Allocs &al, Weights *out) {
  if (w == nullptr) return LLAMA_ERR_INVALID_ARG;
  const void *ptrs[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm, w->w_gate, w->w_up, w->w_down};
  for (const void *p : ptrs) {
    llama_status s = check_ptr(p);
    if (s != LLAMA_OK) return s;
  }
  if (dm.moe()) {
    llama_status s = check_ptr(w->router);
    for (const void *p : {w->shared_gate, w->shared_up, w->shared_down})
      if (s == LLAMA_OK && dm.Fs > 0) s = check_ptr(p);
    if (s != LLAMA_OK) return s;
  }
  const size_t e = dm.esize;
  const size_t dq = (size_t)dm.H * dm.D * dm.d * e, dkv = (size_t)dm.G * dm.D * dm.d * e;
  out->attn_norm = al.alloc(dm.d * e);
  out->ffn_norm = al.alloc(dm.d * e);
  out->wqkv = al.alloc(dq + 2 * dkv);
  out->wo = al.alloc((size_t)dm.d * dm.H * dm.D * e);
  const size_t n_ffn = dm.moe() ? (size_t)dm.E : 1;  // feed-forward weight sets
  out->w_down = al.alloc(n_ffn * dm.d * dm.F * e);
  const bool tc = dm.dtype == LLAMA_BF16;
  if (dm.moe()) {
    out->router = al.alloc((size_t)dm.E_pad * dm.d * e);
    if (dm.Fs > 0) {
      out->shared_gu = al.alloc((size_t)2 * dm.Fs * dm.d * e);
      out->shared_down = al.alloc((size_t)dm.d * dm.Fs * e);
    }
  }
  if (tc) {
    out->w_gu = al.alloc(n_ffn * 2 * dm.F * dm.d * e);
  } else {
    out->w_gate = al.alloc((size_t)dm.F * dm.d * e);
    out->w_up = al.alloc((size_t)dm.F * dm.d * e);
  }
  if (al.failed) return LLAMA_ERR_OOM;
  char *qkv = static_cast<char *>(out->wqkv);
  cudaError_t err = cudaSuccess;
  auto cp = [&](void *dst, const void *src, size_t n) {
    if (err == cudaSuccess) err = cudaMemcpy(dst, src, n, cudaMemcpyDeviceToDevice);
  };
  cp(out->attn_norm, w->attn_norm, dm.d * e);
  cp(out->ffn_norm, w->ffn_norm, dm.d * e);
  if (dm.permute_halves()) {
    if (err == cudaSuccess)
      err = launch_permute_halves_rows((const bf16 *)w->wq, (bf16 *)qkv, dm.H, dm.D, dm.d, nullptr);
    if (err == cudaSuccess)
      err = launch_permute_halves_rows((const bf16 *)w->wk, (bf16 *)(qkv + dq), dm.G, dm.D, dm.d, nullptr);
  } else {
    cp(qkv, w->wq, dq);
    cp(qkv + dq, w->wk, dkv);
  }
  cp(qkv + dq + dkv, w->wv, dkv);
  cp(out->wo, w->wo, (size_t)dm.d * dm.H * dm.D * e);
  cp(out->w_down, w->w_down, n_ffn * dm.d * dm.F * e);
  if (tc) {
    // gate/up rows interleaved in groups of 16 (for experts: one call over all of
    // them, F % 16 == 0 keeps every group inside one expert)
    if (err == cudaSuccess)
      err = launch_interleave_rows((const bf16 *)w->w_gate, (const bf16 *)w->w_up, (bf16 *)out->w_gu,
                                   (int)(n_ffn * dm.F), dm.d, nullptr);
    // RMSNorm gains folded into the consuming projections: (x g) W^T = x (W diag g)^T,
    // so the GEMMs read the raw activations and scale rows by rsqrt(mean(x^2) + eps).
    // Experts read rows the dispatch step has already normalised (gain included).
    if (err == cudaSuccess)
      err = launch_scale_columns((bf16 *)out->wqkv, (const bf16 *)w->attn_norm, dm.QKV, dm.d, nullptr);
    if (err == cudaSuccess && !dm.moe())
      err = launch_scale_columns((bf16 *)out->w_gu, (const bf16 *)w->ffn_norm, 2 * dm.F, dm.d, nullptr);
    if (dm.moe()) {
      if (err == cudaSuccess) err = cudaMemset(out->router, 0, (size_t)dm.E_pad * dm.d * e);
      cp(out->router, w->router, (size_t)dm.E * dm.d * e);
      if (err == cudaSuccess)
        err = launch_scale_columns((bf16 *)out->router, (const bf16 *)w->ffn_norm, dm.E, dm.d, nullptr);
      if (dm.Fs > 0) {
        if (err == cudaSuccess)
          err = launch_interleave_rows((const bf16 *)w->shared_gate, (const bf16 *)w->shared_up,
                                       (bf16 *)out->shared_gu, dm.Fs, dm.d, nullptr);
        if (err == cudaSuccess)
          err = launch_scale_columns((bf16 *)out->shared_gu, (const bf16 *)w->ffn_norm, 2 * dm.Fs, dm.d, nullptr);
        cp(out->shared_down, w->shared_down, (size_t)dm.d * dm.Fs * e);
      }
    }
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
  } else {
    cp(out->w_gate, w->w_gate, (size_t)dm.F * dm.d * e);
    cp(out->w_up, w->w_up, (size_t)dm.F * dm.d * e);
  }
  return err == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA;
}

// Zero the split-K scratch of a workspace.  The GEMM leaves it zero after every
// launch that completes (the last-arriving warp clears what it consumed), so
// this runs at create and after a kernel gave up a bounded wait.
cudaError_t clear_gemm_scratch(const GemmWorkspace &g) {
  cudaError_t e = cudaSuccess;
  if (g.part != nullptr) e = cudaMemset(g.part, 0, g.part_bytes);
  if (e == cudaSuccess && g.counters != nullptr) e = cudaMemset(g.counters, 0, (size_t)g.counter_slots * sizeof(int));
  return e;
}

llama_status alloc_workspace(const Dims &dm, int max_tokens, bool staging, Allocs &al, Workspace *ws) {
  const size_t e = dm.esize, T = (size_t)max_tokens;
  ws->max_tokens = max_tokens;
  if (dm.dtype != LLAMA_BF16) {  // standalone RMSNorm outputs (the bf16 path fuses both norms)
    ws->xn = al.alloc(T * dm.d * e);
    ws->hn = al.alloc(T * dm.d * e);
  }
  if (!dm.fused_qkv_rope())  // unrotated qkv (the bf16 path rotates in the GEMM epilogue)
    ws->qkv = al.alloc(T * dm.QKV * e);
  ws->q = al.alloc(T * dm.H * dm.D * e);
  ws->o = al.alloc(T * dm.H * dm.D * e);
  ws->h = al.alloc(T * dm.d * e);
  if (!dm.moe()) ws->act = al.alloc(T * dm.F * e);
  if (dm.moe()) {
    const size_t Tk = T * dm.topk;
    ws->logits = (float *)al.alloc(T * dm.E_pad * sizeof(float));
    ws->route_w = (float *)al.alloc(Tk * sizeof(float));
    ws->route_ids = (int *)al.alloc(Tk * sizeof(int));
    ws->route_pos = (int *)al.alloc(Tk * sizeof(int));
    ws->counts = (int *)al.alloc((size_t)dm.E * sizeof(int));
    ws->offsets = (int *)al.alloc((size_t)(dm.E + 1) * sizeof(int));
    ws->fill = (int *)al.alloc((size_t)dm.E * sizeof(int));
    ws->xin_e = al.alloc(Tk * dm.d * e);
    ws->act_e = al.alloc(Tk * dm.F * e);
    ws->y_e = al.alloc(Tk * dm.d * e);
    if (dm.Fs > 0) {
      ws->act_s = al.alloc(T * dm.Fs * e);
      ws->hs = al.alloc(T * dm.d * e);
    }
  }
  if (staging) {
    ws->xin = al.alloc(T * dm.d * e);
    ws->yout = al.alloc(T * dm.d * e);
  }
  if (dm.dtype == LLAMA_BF16) {
    const size_t bytes = attn_decode_scratch_bytes(max_tokens, dm.H, dm.D, dm.max_seq);
    ws->attn.partial = al.alloc(bytes);
    ws->attn.bytes = bytes;
    ws->attn.item_counters = (int *)al.alloc(2 * sizeof(int));
    ws->gemm.part_bytes = gemm_splitk_part_bytes();
    ws->gemm.part = (float *)al.alloc(ws->gemm.part_bytes);
    ws->gemm.counter_slots = gemm_splitk_counter_slots();
    ws->gemm.counters = (int *)al.alloc((size_t)ws->gemm.counter_slots * sizeof(int));
    ws->ss_x = (float *)al.alloc(T * sizeof(float));
    ws->ss_h = (float *)al.alloc(T * sizeof(float));
    ws->ss_x2 = (float *)al.alloc(T * sizeof(float));
    ws->fused_sync = (unsigned *)al.alloc(2 * sizeof(unsigned));
  }
  if (al.failed) return LLAMA_ERR_OOM;
  if (clear_gemm_scratch(ws->gemm) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (ws->attn.item_counters != nullptr && cudaMemset(ws->attn.item_counters, 0, 2 * sizeof(int)) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  if (dm.moe() && (cudaMemset(ws->counts, 0, (size_t)dm.E * sizeof(int)) != cudaSuccess ||
                   cudaMemset(ws->fill, 0, (size_t)dm.E * sizeof(int)) != cudaSuccess))
    return LLAMA_ERR_CUDA;
  return LLAMA_OK;
}

#define LAUNCH(expr)                                 \
  do {                                               \
    cudaError_t _e = (expr);                         \
    if (_e != cudaSuccess) {                         \
      note_cuda_error(_e);                           \
      return LLAMA_ERR_CUDA;                         \
    }                                                \
  } while (0)

// The handle's cos/sin table: grouped for the GEMM epilogue when that applies the
// rotation (bf16, D % 32 == 0), else row-major for rope_kv_kernel.
cudaError_t launch_rope_table_any(const Dims &dm, float2 *table) {
  return dm.fused_qkv_rope() ? launch_rope_table_grouped(table, dm.max_seq, dm.D, dm.theta, dm.rope_scaling, nullptr)
                             : launch_rope_table(table, dm.max_seq, dm.D, dm.theta, dm.rope_scaling, nullptr);
}

template <typename T>
llama_status forward_simt(const Dims &dm, const Weights &w, const Workspace &ws, const float2 *rope, const T *x,
                          T *y, int B, int S, int start_pos, const llama_kv_cache *kv, cudaStream_t st) {
  const int M = B * S;
  T *xn = (T *)ws.xn, *qkv = (T *)ws.qkv, *q = (T *)ws.q, *o = (T *)ws.o, *h = (T *)ws.h, *act = (T *)ws.act,
    *hn = (T *)ws.hn;
  LAUNCH(launch_rmsnorm<T>(x, (const T *)w.attn_norm, xn, M, dm.d, dm.eps, st));
  LAUNCH(launch_gemm_simt<T>(xn, (const T *)w.wqkv, nullptr, nullptr, qkv, M, dm.QKV, dm.d, EPI_STORE, st));
  LAUNCH(launch_rope_kv<T>(qkv, q, (T *)kv->k, (T *)kv->v, rope, B, S, start_pos, dm.H, dm.G, dm.D,
                           kv->max_seq_len, dm.rope_halves, st));
  LAUNCH(launch_attention_simt<T>(q, (const T *)kv->k, (const T *)kv->v, o, B, S, start_pos, dm.H, dm.G, dm.D,
                                  kv->max_seq_len, st));
  LAUNCH(launch_gemm_simt<T>(o, (const T *)w.wo, nullptr, x, h, M, dm.d, dm.H * dm.D, EPI_RESIDUAL, st));
  LAUNCH(launch_rmsnorm<T>(h, (const T *)w.ffn_norm, hn, M, dm.d, dm.eps, st));
  LAUNCH(launch_gemm_simt<T>(hn, (const T *)w.w_gate, (const T *)w.w_up, nullptr, act, M, dm.F, dm.d, EPI_SWIGLU,
                             st));
  LAUNCH(launch_gemm_simt<T>(act, (const T *)w.w_down, nullptr, h, y, M, dm.d, dm.F, EPI_RESIDUAL, st));
  return LLAMA_OK;
}

// Mixture-of-experts feed-forward of a bf16 block ("Llama 4 From Scratch", MoE):
// router logits (GEMM with the ffn-norm row scale), top-k routing, per-expert
// row offsets, dispatch of the normalised rows, the experts' SwiGLU as two
// grouped GEMMs over those row ranges, the shared expert as the dense fused
// path (its down projection adds the residual), and the weighted combine.
llama_status forward_moe(const Dims &dm, const Weights &w, const Workspace &ws, const bf16 *h, bf16 *y, int M,
                         const RowNorm &norm_h, int *status, Profiler &pf, cudaStream_t st) {
  const int k = dm.topk, Mk = M * dm.topk;
  bf16 *xin = (bf16 *)ws.xin_e, *act = (bf16 *)ws.act_e, *ye = (bf16 *)ws.y_e;
  pf.mark(5, 0, st);  // ffn_norm slot: routing and dispatch
  LAUNCH(launch_gemm_tc(h, (const bf16 *)w.router, nullptr, ws.logits, M, dm.E_pad, dm.d, EPI_F32OUT_ROWSCALE,
                        status, st, &ws.gemm, &norm_h, nullptr, true));
  LAUNCH(launch_moe_topk(ws.logits, dm.E_pad, M, dm.E, k, ws.route_ids, ws.route_w, ws.counts, st));
  LAUNCH(launch_moe_offsets(ws.counts, ws.offsets, ws.fill, dm.E, st));
  LAUNCH(launch_moe_dispatch(h, ws.ss_h, (const bf16 *)w.ffn_norm, dm.eps, M, dm.d, k, ws.route_ids, ws.offsets,
                             ws.fill, ws.route_pos, xin, st));
  pf.mark(5, 1, st);
  pf.mark(6, 0, st);  // gate/up slot: experts and shared expert
  LAUNCH(launch_gemm_grouped(xin, (const bf16 *)w.w_gu, act, Mk, 2 * dm.F, dm.d, dm.E, ws.offsets, EPI_SWIGLU,
                             status, st));
  if (dm.Fs > 0)
    LAUNCH(launch_gemm_tc(h, (const bf16 *)w.shared_gu, nullptr, ws.act_s, M, 2 * dm.Fs, dm.d, EPI_SWIGLU_ROWSCALE,
                          status, st, &ws.gemm, &norm_h, nullptr, true));
  pf.mark(6, 1, st);
  pf.mark(7, 0, st);  // down slot: experts, shared expert (+ residual), combine
  LAUNCH(launch_gemm_grouped(act, (const bf16 *)w.w_down, ye, Mk, dm.d, dm.F, dm.E, ws.offsets, EPI_STORE, status,
                             st));
  const bf16 *base = h;
  if (dm.Fs > 0) {
    LAUNCH(launch_gemm_tc((const bf16 *)ws.act_s, (const bf16 *)w.shared_down, h, ws.hs, M, dm.d, dm.Fs,
                          EPI_RESIDUAL, status, st, &ws.gemm, nullptr, nullptr, true));
    base = (const bf16 *)ws.hs;
  }
  LAUNCH(launch_moe_combine(base, ye, ws.route_pos, ws.route_w, M, dm.d, k, y, st));
  pf.mark(7, 1, st);
  return LLAMA_OK;
}

// A decode step this handle may run as the fused kernel (decode_fused.cu).
bool fused_decode_eligible(const Dims &dm, int S) {
  return S == 1 && dm.dtype == LLAMA_BF16 && !dm.moe() && dm.fused_qkv_rope() &&
         attn_decode_tc_supported(dm.H, dm.G, dm.D);
}

llama_status forward_decode_fused(const Dims &dm, const Weights &w, const Workspace &ws, const float2 *rope,
                                  const bf16 *x, bf16 *y, int B, int start_pos, const llama_kv_cache *kv, int *status,
                                  cudaStream_t st) {
  DecodeFusedParams p;
  p.x = x;
  p.y = y;
  p.wqkv = (const bf16 *)w.wqkv;
  p.wo = (const bf16 *)w.wo;
  p.w_gu = (const bf16 *)w.w_gu;
  p.w_down = (const bf16 *)w.w_down;
  p.q = (bf16 *)ws.q;
  p.o = (bf16 *)ws.o;
  p.h = (bf16 *)ws.h;
  p.act = (bf16 *)ws.act;
  p.ss_x = ws.ss_x;
  p.ss_h = ws.ss_h;
  p.rope = rope;
  p.rope_seq = dm.max_seq;
  p.kc = (bf16 *)kv->k;
  p.vc = (bf16 *)kv->v;
  p.cache_seq = kv->max_seq_len;
  p.B = B;
  p.start_pos = start_pos;
  p.d = dm.d;
  p.H = dm.H;
  p.G = dm.G;
  p.D = dm.D;
  p.F = dm.F;
  p.halves = dm.rope_halves;
  p.eps = dm.eps;
  p.gemm = ws.gemm;
  p.attn = ws.attn;
  p.sync = ws.fused_sync;
  p.status = status;
  LAUNCH(launch_decode_block_fused(p, st));
  return LLAMA_OK;
}

// Row statistics handed from one block of a stack to the next: the down
// projection's epilogue sums the squares of the rows of y it stores, which are
// the next block's attention-norm statistics, so the next block skips its
// statistics pass.  The two input buffers alternate between blocks.
struct LayerStats {
  float *in = nullptr;    // sums of squares of x's rows, already accumulated (null: compute them here)
  float *next = nullptr;  // accumulate the sums of squares of y's rows here, zero on entry (null: don't)
};

llama_status forward_tc(const Dims &dm, const Weights &w, const Workspace &ws, const float2 *rope, const bf16 *x,
                        bf16 *y, int B, int S, int start_pos, const llama_kv_cache *kv, int *status, Profiler *prof,
                        cudaStream_t st, const LayerStats *ls = nullptr) {
  if (ws.decode_mode == LLAMA_DECODE_FUSED && fused_decode_eligible(dm, S))
    return forward_decode_fused(dm, w, ws, rope, x, y, B, start_pos, kv, status, st);
  const int M = B * S;
  bf16 *qkv = (bf16 *)ws.qkv, *q = (bf16 *)ws.q, *o = (bf16 *)ws.o, *h = (bf16 *)ws.h, *act = (bf16 *)ws.act;
  bf16 *kc = (bf16 *)kv->k, *vc = (bf16 *)kv->v;
  Profiler none;
  Profiler &pf = prof != nullptr ? *prof : none;
  pf.begin_forward();
  // attention_norm statistics; the normalisation itself happens in the QKV GEMM
  pf.mark(0, 0, st);
  const bool stats_ready = ls != nullptr && ls->in != nullptr;
  float *ss_x = stats_ready ? ls->in : ws.ss_x;
  if (!stats_ready)  // also clears the accumulators this forward adds into
    LAUNCH(launch_row_sqsum(x, ws.ss_x, ws.ss_h, M, dm.d, st, ls != nullptr ? ls->next : nullptr));
  pf.mark(0, 1, st);
  RowNorm norm_x;
  norm_x.ss_in = ss_x;
  norm_x.eps = dm.eps;
  norm_x.d = dm.d;
  if (dm.fused_qkv_rope()) {
    // QKV projection, RoPE and the cache write in one GEMM epilogue
    QkvScatter sc;
    sc.table = rope;
    sc.table_seq = dm.max_seq;
    sc.q = q;
    sc.kc = kc;
    sc.vc = vc;
    sc.S = S;
    sc.start_pos = start_pos;
    sc.H = dm.H;
    sc.G = dm.G;
    sc.D = dm.D;
    sc.cache_seq = kv->max_seq_len;
    sc.halves = dm.rope_halves;
    pf.mark(1, 0, st);
    LAUNCH(launch_gemm_tc(x, (const bf16 *)w.wqkv, nullptr, nullptr, M, dm.QKV, dm.d, EPI_QKV_ROPE, status, st,
                          &ws.gemm, &norm_x, &sc, true));
    pf.mark(1, 1, st);
    pf.mark(2, 0, st);  // RoPE + KV write: fused into the QKV epilogue
    pf.mark(2, 1, st);
  } else {
    pf.mark(1, 0, st);
    LAUNCH(launch_gemm_tc(x, (const bf16 *)w.wqkv, nullptr, qkv, M, dm.QKV, dm.d, EPI_STORE_ROWSCALE, status, st,
                          &ws.gemm, &norm_x, nullptr, true));
    pf.mark(1, 1, st);
    pf.mark(2, 0, st);
    LAUNCH(launch_rope_kv<bf16>(qkv, q, kc, vc, rope, B, S, start_pos, dm.H, dm.G, dm.D, kv->max_seq_len,
                                dm.rope_halves, st));
    pf.mark(2, 1, st);
  }
  pf.mark(3, 0, st);
  LAUNCH(launch_attention(q, kc, vc, o, B, S, start_pos, dm.H, dm.G, dm.D, kv->max_seq_len, ws.attn, status, st));
  pf.mark(3, 1, st);
  // h = x + o Wo^T; the epilogue also accumulates the ffn_norm statistics of h
  RowNorm norm_h;
  norm_h.ss_in = ws.ss_h;
  norm_h.ss_out = ws.ss_h;
  norm_h.eps = dm.eps;
  norm_h.d = dm.d;
  pf.mark(4, 0, st);
  LAUNCH(launch_gemm_tc(o, (const bf16 *)w.wo, x, h, M, dm.d, dm.H * dm.D, EPI_RESIDUAL_SQSUM, status, st, &ws.gemm,
                        &norm_h, nullptr, true));
  pf.mark(4, 1, st);
  if (dm.moe()) return forward_moe(dm, w, ws, h, y, M, norm_h, status, pf, st);
  pf.mark(5, 0, st);  // ffn_norm: fused into the O and gate/up GEMM epilogues
  pf.mark(5, 1, st);
  pf.mark(6, 0, st);
  LAUNCH(launch_gemm_tc(h, (const bf16 *)w.w_gu, nullptr, act, M, 2 * dm.F, dm.d, EPI_SWIGLU_ROWSCALE, status, st,
                        &ws.gemm, &norm_h, nullptr, true));
  pf.mark(6, 1, st);
  pf.mark(7, 0, st);
  if (ls != nullptr && ls->next != nullptr) {
    // y's statistics for the next block; this block's input statistics and the
    // ffn-norm accumulator are read by now and are cleared for the blocks after
    RowNorm norm_y;
    norm_y.ss_out = ls->next;
    norm_y.zero_a = ss_x;
    norm_y.zero_b = ws.ss_h;
    norm_y.eps = dm.eps;
    norm_y.d = dm.d;
    LAUNCH(launch_gemm_tc(act, (const bf16 *)w.w_down, h, y, M, dm.d, dm.F, EPI_RESIDUAL_SQSUM, status, st,
                          &ws.gemm, &norm_y, nullptr, true));
  } else {
    LAUNCH(launch_gemm_tc(act, (const bf16 *)w.w_down, h, y, M, dm.d, dm.F, EPI_RESIDUAL, status, st, &ws.gemm,
                          nullptr, nullptr, true));
  }
  pf.mark(7, 1, st);
  return LLAMA_OK;
}

llama_status forward_any(const Dims &dm, const Weights &w, const Workspace &ws, const float2 *rope, const void *x,
                         void *y, int B, int S, int start_pos, const llama_kv_cache *kv, int *status,
                         cudaStream_t st, Profiler *prof = nullptr, const LayerStats *ls = nullptr) {
  if (dm.dtype == LLAMA_BF16)
    return forward_tc(dm, w, ws, rope, (const bf16 *)x, (bf16 *)y, B, S, start_pos, kv, status, prof, st, ls);
  return forward_simt<float>(dm, w, ws, rope, (const float *)x, (float *)y, B, S, start_pos, kv, st);
}

llama_status validate_call(const Dims &dm, int max_tokens, int B, int S, int start_pos, const llama_kv_cache *kv) {
  if (kv == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || start_pos < 0) return LLAMA_ERR_INVALID_ARG;
  if ((long long)B * S > max_tokens) return LLAMA_ERR_RANGE;
  if (B > kv->max_batch) return LLAMA_ERR_RANGE;
  if ((long long)start_pos + S > dm.max_seq || (long long)start_pos + S > kv->max_seq_len) return LLAMA_ERR_RANGE;
  llama_status s = check_ptr(kv->k);
  if (s != LLAMA_OK) return s;
  return check_ptr(kv->v);
}

llama_status read_status(int *dev_status, int device, const Workspace *ws, const Dims *dm) {
  const GemmWorkspace *scratch = ws != nullptr ? &ws->gemm : nullptr;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return LLAMA_ERR_CUDA;
  int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&v, dev_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(dev_status, 0, sizeof(int));
  if (e == cudaSuccess && v != 0 && v != DEV_BAD_TOKEN && scratch != nullptr) {
    e = clear_gemm_scratch(*scratch);
    if (e == cudaSuccess && ws->attn.item_counters != nullptr)
      e = cudaMemset(ws->attn.item_counters, 0, 2 * sizeof(int));
    if (e == cudaSuccess && dm != nullptr && dm->moe()) e = cudaMemset(ws->counts, 0, (size_t)dm->E * sizeof(int));
    if (e == cudaSuccess && dm != nullptr && dm->moe()) e = cudaMemset(ws->fill, 0, (size_t)dm->E * sizeof(int));
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) return LLAMA_ERR_CUDA;
  if (v == 0) return LLAMA_OK;
  return v == DEV_BAD_TOKEN ? LLAMA_ERR_RANGE : LLAMA_ERR_DEVICE_TIMEOUT;
}

}  // namespace

struct llama_block {
  Dims dm;
  int device = 0;
  Allocs al;
  Weights w;
  Workspace ws;
  float2 *rope = nullptr;
  int *status = nullptr;
  Profiler prof;
};

struct llama_stack {
  Dims dm;
  int device = 0, n_layers = 0, vocab = 0;
  Allocs al;
  std::vector<Weights> layers;
  Workspace ws;
  float2 *rope = nullptr;
  int *status = nullptr;
  void *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
  void *x0 = nullptr, *x1 = nullptr, *xn = nullptr;
  int32_t *next_tok = nullptr;  // greedy decoding: the ids fed to the next step [max_tokens]
};

extern "C" {

llama_status llama_block_create(const llama_config *cfg, const llama_block_weights *w, int32_t max_tokens,
                                llama_block **out) {
  if (out == nullptr) return LLAMA_ERR_INVALID_ARG;
  *out = nullptr;
  Dims dm;
  llama_status s = validate_config(cfg, &dm);
  if (s != LLAMA_OK) return s;
  if (max_tokens <= 0) return LLAMA_ERR_INVALID_ARG;
  llama_block *b = new (std::nothrow) llama_block();
  if (b == nullptr) return LLAMA_ERR_OOM;
  b->dm = dm;
  cudaGetDevice(&b->device);
  s = copy_weights(dm, w, b->al, &b->w);
  if (s == LLAMA_OK) s = alloc_workspace(dm, max_tokens, true, b->al, &b->ws);
  if (s == LLAMA_OK) {
    b->rope = (float2 *)b->al.alloc((size_t)dm.max_seq * (dm.D / 2) * sizeof(float2));
    b->status = (int *)b->al.alloc(sizeof(DeviceStatus));
    if (b->al.failed) s = LLAMA_ERR_OOM;
  }
  if (s == LLAMA_OK) {
    if (launch_rope_table_any(dm, b->rope) != cudaSuccess ||
        cudaMemset(b->status, 0, sizeof(DeviceStatus)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      s = LLAMA_ERR_CUDA;
  }
  if (s != LLAMA_OK) {
    b->al.free_all();
    delete b;
    return s;
  }
  *out = b;
  return LLAMA_OK;
}

llama_status llama_block_forward(llama_block *blk, const void *x, void *y, int32_t B, int32_t S, int32_t start_pos,
                                 const llama_kv_cache *kv, llama_stream stream) {
  if (blk == nullptr) return LLAMA_ERR_INVALID_ARG;
  llama_status s = check_ptr(x);
  if (s == LLAMA_OK) s = check_ptr(y);
  if (s == LLAMA_OK) s = validate_call(blk->dm, blk->ws.max_tokens, B, S, start_pos, kv);
  if (s != LLAMA_OK) return s;
  s = forward_any(blk->dm, blk->w, blk->ws, blk->rope, x, y, B, S, start_pos, kv, blk->status, (cudaStream_t)stream,
                  &blk->prof);
  if (s == LLAMA_OK) blk->ws.last_tokens = B * S;
  return s;
}

llama_status llama_block_forward_host(llama_block *blk, const void *x_host, void *y_host, int32_t B, int32_t S,
                                      int32_t start_pos, const llama_kv_cache *kv, llama_stream stream) {
  if (blk == nullptr || x_host == nullptr || y_host == nullptr) return LLAMA_ERR_INVALID_ARG;
  llama_status s = validate_call(blk->dm, blk->ws.max_tokens, B, S, start_pos, kv);
  if (s != LLAMA_OK) return s;
  const size_t bytes = (size_t)B * S * blk->dm.d * blk->dm.esize;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(blk->ws.xin, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return LLAMA_ERR_CUDA;
  s = forward_any(blk->dm, blk->w, blk->ws, blk->rope, blk->ws.xin, blk->ws.yout, B, S, start_pos, kv,
                  blk->status, st, &blk->prof);
  if (s != LLAMA_OK) return s;
  blk->ws.last_tokens = B * S;
  if (cudaMemcpyAsync(y_host, blk->ws.yout, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return LLAMA_ERR_CUDA;
  return LLAMA_OK;
}

void llama_block_destroy(llama_block *blk) {
  if (blk == nullptr) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(blk->device);
  cudaDeviceSynchronize();
  blk->prof.release();
  blk->al.free_all();
  cudaSetDevice(prev);
  delete blk;
}

llama_status llama_block_profile_enable(llama_block *blk, int32_t max_forwards) {
  if (blk == nullptr || max_forwards <= 0) return LLAMA_ERR_INVALID_ARG;
  blk->prof.release();
  blk->prof.ev.resize((size_t)max_forwards * LLAMA_PROFILE_STEPS * 2);
  blk->prof.launched.assign((size_t)max_forwards * LLAMA_PROFILE_STEPS, 0);
  for (cudaEvent_t &e : blk->prof.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      blk->prof.release();
      return LLAMA_ERR_CUDA;
    }
  }
  blk->prof.max_forwards = max_forwards;
  blk->prof.used = 0;
  blk->prof.on = true;
  return LLAMA_OK;
}

llama_status llama_block_profile_disable(llama_block *blk) {
  if (blk == nullptr) return LLAMA_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  blk->prof.release();
  return LLAMA_OK;
}

llama_status llama_block_profile_read(llama_block *blk, int32_t *launches, float *total_ms) {
  if (blk == nullptr || launches == nullptr || total_ms == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return LLAMA_ERR_CUDA;
  for (int s = 0; s < LLAMA_PROFILE_STEPS; ++s) {
    launches[s] = 0;
    total_ms[s] = 0.f;
  }
  Profiler &p = blk->prof;
  for (int f = 0; f < p.used; ++f)
    for (int s = 0; s < LLAMA_PROFILE_STEPS; ++s) {
      float ms = 0.f;
      cudaEvent_t *e = &p.ev[((size_t)f * LLAMA_PROFILE_STEPS + s) * 2];
      if (!p.launched[(size_t)f * LLAMA_PROFILE_STEPS + s]) continue;  // fused into another step's kernel
      if (cudaEventElapsedTime(&ms, e[0], e[1]) == cudaSuccess) {
        launches[s] += 1;
        total_ms[s] += ms;
      } else {
        cudaGetLastError();
      }
    }
  p.used = 0;
  return LLAMA_OK;
}

llama_status llama_block_moe_routing(llama_block *blk, int32_t *ids, float *weights, llama_stream stream) {
  if (blk == nullptr || !blk->dm.moe() || blk->ws.last_tokens <= 0) return LLAMA_ERR_INVALID_ARG;
  llama_status s = check_ptr(ids);
  if (s == LLAMA_OK) s = check_ptr(weights);
  if (s != LLAMA_OK) return s;
  const size_t n = (size_t)blk->ws.last_tokens * blk->dm.topk;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(ids, blk->ws.route_ids, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(weights, blk->ws.route_w, n * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  return LLAMA_OK;
}

const char *llama_profile_step_name(int32_t step) {
  static const char *names[LLAMA_PROFILE_STEPS] = {"attention_norm", "qkv_projection", "rope_kv_write",
                                                   "attention", "o_projection_residual", "ffn_norm",
                                                   "gate_up_swiglu", "down_projection_residual"};
  return (step >= 0 && step < LLAMA_PROFILE_STEPS) ? names[step] : "unknown";
}

static llama_status set_decode_mode(Workspace &ws, int device, int32_t mode) {
  if (mode != LLAMA_DECODE_KERNELS && mode != LLAMA_DECODE_FUSED) return LLAMA_ERR_INVALID_ARG;
  if (mode == LLAMA_DECODE_FUSED) {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return LLAMA_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return LLAMA_ERR_CUDA;
    const bool ok = ws.fused_sync != nullptr && decode_fused_available();
    if (prev != device) cudaSetDevice(prev);
    if (!ok) return LLAMA_ERR_UNSUPPORTED;
  }
  ws.decode_mode = mode;
  return LLAMA_OK;
}

llama_status llama_block_set_decode_mode(llama_block *blk, int32_t mode) {
  if (blk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return set_decode_mode(blk->ws, blk->device, mode);
}

llama_status llama_stack_set_decode_mode(llama_stack *stk, int32_t mode) {
  if (stk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return set_decode_mode(stk->ws, stk->device, mode);
}

// Writes the wait budget (cycles, 0 = the default) of a handle's status block.
static llama_status set_wait_budget(int *dev_status, int device, int64_t cycles) {
  if (cycles < 0) return LLAMA_ERR_INVALID_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return LLAMA_ERR_CUDA;
  const long long v = cycles;
  DeviceStatus *blk = reinterpret_cast<DeviceStatus *>(dev_status);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&blk->wait_budget, &v, sizeof(v), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return LLAMA_ERR_CUDA;
  }
  return LLAMA_OK;
}

llama_status llama_block_set_wait_budget(llama_block *blk, int64_t cycles) {
  if (blk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return set_wait_budget(blk->status, blk->device, cycles);
}

llama_status llama_stack_set_wait_budget(llama_stack *stk, int64_t cycles) {
  if (stk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return set_wait_budget(stk->status, stk->device, cycles);
}

llama_status llama_block_device_status(llama_block *blk) {
  if (blk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return read_status(blk->status, blk->device, &blk->ws, &blk->dm);
}

llama_status llama_stack_create(const llama_config *cfg, int32_t n_layers, int32_t vocab, const void *embed,
                                const llama_block_weights *layers, const void *final_norm, const void *lm_head,
                                int32_t max_tokens, llama_stack **out) {
  if (out == nullptr) return LLAMA_ERR_INVALID_ARG;
  *out = nullptr;
  Dims dm;
  llama_status s = validate_config(cfg, &dm);
  if (s != LLAMA_OK) return s;
  if (n_layers < 0 || vocab <= 0 || max_tokens <= 0 || (n_layers > 0 && layers == nullptr))
    return LLAMA_ERR_INVALID_ARG;
  for (const void *p : {embed, final_norm, lm_head}) {
    s = check_ptr(p);
    if (s != LLAMA_OK) return s;
  }
  llama_stack *k = new (std::nothrow) llama_stack();
  if (k == nullptr) return LLAMA_ERR_OOM;
  k->dm = dm;
  k->n_layers = n_layers;
  k->vocab = vocab;
  cudaGetDevice(&k->device);
  k->layers.resize(n_layers);
  for (int l = 0; l < n_layers && s == LLAMA_OK; ++l) s = copy_weights(dm, &layers[l], k->al, &k->layers[l]);
  if (s == LLAMA_OK) s = alloc_workspace(dm, max_tokens, false, k->al, &k->ws);
  const size_t e = dm.esize;
  if (s == LLAMA_OK) {
    k->embed = k->al.alloc((size_t)vocab * dm.d * e);
    k->lm_head = k->al.alloc((size_t)vocab * dm.d * e);
    k->final_norm = k->al.alloc(dm.d * e);
    k->x0 = k->al.alloc((size_t)max_tokens * dm.d * e);
    k->x1 = k->al.alloc((size_t)max_tokens * dm.d * e);
    k->xn = k->al.alloc((size_t)max_tokens * dm.d * e);
    k->next_tok = (int32_t *)k->al.alloc((size_t)max_tokens * sizeof(int32_t));
    k->rope = (float2 *)k->al.alloc((size_t)dm.max_seq * (dm.D / 2) * sizeof(float2));
    k->status = (int *)k->al.alloc(sizeof(DeviceStatus));
    if (k->al.failed) s = LLAMA_ERR_OOM;
  }
  if (s == LLAMA_OK) {
    cudaError_t err = cudaMemcpy(k->embed, embed, (size_t)vocab * dm.d * e, cudaMemcpyDeviceToDevice);
    if (err == cudaSuccess) err = cudaMemcpy(k->lm_head, lm_head, (size_t)vocab * dm.d * e, cudaMemcpyDeviceToDevice);
    if (err == cudaSuccess) err = cudaMemcpy(k->final_norm, final_norm, dm.d * e, cudaMemcpyDeviceToDevice);
    if (err == cudaSuccess) err = launch_rope_table_any(dm, k->rope);
    if (err == cudaSuccess) err = cudaMemset(k->status, 0, sizeof(DeviceStatus));
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
    if (err != cudaSuccess) s = LLAMA_ERR_CUDA;
  }
  if (s != LLAMA_OK) {
    k->al.free_all();
    delete k;
    return s;
  }
  *out = k;
  return LLAMA_OK;
}

}  // extern "C"

namespace {

// Embedding gather and the N blocks; returns the buffer holding the last
// block's output [B*S][d] in *hidden.
llama_status stack_layers(llama_stack *stk, const int32_t *tokens, int B, int S, int start_pos,
                          const llama_kv_cache *kv, cudaStream_t st, void **hidden) {
  const Dims &dm = stk->dm;
  const int M = B * S;
  void *cur = stk->x0, *nxt = stk->x1;
  if (dm.dtype == LLAMA_BF16)
    LAUNCH(launch_embed<bf16>(tokens, (const bf16 *)stk->embed, (bf16 *)cur, M, dm.d, stk->vocab, stk->status, st));
  else
    LAUNCH(launch_embed<float>(tokens, (const float *)stk->embed, (float *)cur, M, dm.d, stk->vocab, stk->status, st));
  // dense bf16 blocks hand their row statistics on (LayerStats); not the
  // mixture-of-experts feed-forward nor the fused decode kernel
  const bool chain = dm.dtype == LLAMA_BF16 && !dm.moe() &&
                     !(stk->ws.decode_mode == LLAMA_DECODE_FUSED && fused_decode_eligible(dm, S));
  float *stats[2] = {stk->ws.ss_x, stk->ws.ss_x2};
  for (int l = 0; l < stk->n_layers; ++l) {
    LayerStats ls;
    if (chain) {
      ls.in = l == 0 ? nullptr : stats[l & 1];
      ls.next = l + 1 < stk->n_layers ? stats[(l + 1) & 1] : nullptr;
    }
    llama_status s = forward_any(dm, stk->layers[l], stk->ws, stk->rope, cur, nxt, B, S, start_pos, &kv[l],
                                 stk->status, st, nullptr, chain ? &ls : nullptr);
    if (s != LLAMA_OK) return s;
    void *t = cur;
    cur = nxt;
    nxt = t;
  }
  *hidden = cur;
  return LLAMA_OK;
}

// Final RMSNorm and the LM head over `rows` rows of `hidden`: logits [rows][vocab] fp32.
llama_status stack_head(llama_stack *stk, const void *hidden, int rows, float *logits, cudaStream_t st) {
  const Dims &dm = stk->dm;
  if (dm.dtype == LLAMA_BF16) {
    LAUNCH(launch_rmsnorm<bf16>((const bf16 *)hidden, (const bf16 *)stk->final_norm, (bf16 *)stk->xn, rows, dm.d,
                                dm.eps, st));
    LAUNCH(launch_gemm_tc((const bf16 *)stk->xn, (const bf16 *)stk->lm_head, nullptr, logits, rows, stk->vocab, dm.d,
                          EPI_F32OUT, stk->status, st, &stk->ws.gemm, nullptr, nullptr, true));
  } else {
    LAUNCH(launch_rmsnorm<float>((const float *)hidden, (const float *)stk->final_norm, (float *)stk->xn, rows, dm.d,
                                 dm.eps, st));
    LAUNCH(launch_gemm_simt<float>((const float *)stk->xn, (const float *)stk->lm_head, nullptr, nullptr, logits,
                                   rows, stk->vocab, dm.d, EPI_F32OUT, st));
  }
  return LLAMA_OK;
}

}  // namespace

extern "C" {

llama_status llama_stack_forward(llama_stack *stk, const int32_t *tokens, int32_t B, int32_t S, int32_t start_pos,
                                 const llama_kv_cache *kv, float *logits, llama_stream stream) {
  if (stk == nullptr || (kv == nullptr && stk->n_layers > 0)) return LLAMA_ERR_INVALID_ARG;
  llama_status s = check_ptr(tokens);
  if (s == LLAMA_OK) s = check_ptr(logits);
  if (s != LLAMA_OK) return s;
  if (B <= 0 || S <= 0 || start_pos < 0) return LLAMA_ERR_INVALID_ARG;
  if ((long long)B * S > stk->ws.max_tokens || (long long)start_pos + S > stk->dm.max_seq) return LLAMA_ERR_RANGE;
  for (int l = 0; l < stk->n_layers; ++l) {
    s = validate_call(stk->dm, stk->ws.max_tokens, B, S, start_pos, &kv[l]);
    if (s != LLAMA_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  void *hidden = nullptr;
  s = stack_layers(stk, tokens, B, S, start_pos, kv, st, &hidden);
  if (s != LLAMA_OK) return s;
  return stack_head(stk, hidden, B * S, logits, st);
}

llama_status llama_stack_generate(llama_stack *stk, const int32_t *prompt, int32_t B, int32_t S_prompt,
                                  int32_t start_pos, int32_t n_new, const llama_kv_cache *kv, int32_t *out_tokens,
                                  float *logits, llama_stream stream) {
  if (stk == nullptr || (kv == nullptr && stk->n_layers > 0)) return LLAMA_ERR_INVALID_ARG;
  llama_status s = check_ptr(prompt);
  if (s == LLAMA_OK) s = check_ptr(out_tokens);
  if (s == LLAMA_OK) s = check_ptr(logits);
  if (s != LLAMA_OK) return s;
  if (B <= 0 || S_prompt <= 0 || start_pos < 0 || n_new <= 0) return LLAMA_ERR_INVALID_ARG;
  // positions start_pos .. start_pos + S_prompt + n_new - 2 are run (the last pick is not fed back)
  const long long last_pos = (long long)start_pos + S_prompt + n_new - 2;
  if ((long long)B * S_prompt > stk->ws.max_tokens || last_pos + 1 > stk->dm.max_seq) return LLAMA_ERR_RANGE;
  for (int l = 0; l < stk->n_layers; ++l) {
    s = validate_call(stk->dm, stk->ws.max_tokens, B, S_prompt, start_pos, &kv[l]);
    if (s == LLAMA_OK && last_pos + 1 > kv[l].max_seq_len) s = LLAMA_ERR_RANGE;
    if (s != LLAMA_OK) return s;
  }
  const Dims &dm = stk->dm;
  cudaStream_t st = (cudaStream_t)stream;
  int pos = start_pos;
  for (int i = 0; i < n_new; ++i) {
    const int S = i == 0 ? S_prompt : 1;
    void *hidden = nullptr;
    s = stack_layers(stk, i == 0 ? prompt : stk->next_tok, B, S, pos, kv, st, &hidden);
    if (s != LLAMA_OK) return s;
    const void *last = hidden;
    if (S > 1) {  // the last position of each sequence, into the free ping-pong buffer
      void *dst = hidden == stk->x0 ? stk->x1 : stk->x0;
      if (dm.dtype == LLAMA_BF16)
        LAUNCH(launch_gather_last_rows<bf16>((const bf16 *)hidden, (bf16 *)dst, B, S, dm.d, st));
      else
        LAUNCH(launch_gather_last_rows<float>((const float *)hidden, (float *)dst, B, S, dm.d, st));
      last = dst;
    }
    s = stack_head(stk, last, B, logits, st);
    if (s != LLAMA_OK) return s;
    LAUNCH(launch_argmax_rows(logits, B, stk->vocab, out_tokens + i, n_new, stk->next_tok, st));
    pos += S;
  }
  return LLAMA_OK;
}

void llama_stack_destroy(llama_stack *stk) {
  if (stk == nullptr) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(stk->device);
  cudaDeviceSynchronize();
  stk->al.free_all();
  cudaSetDevice(prev);
  delete stk;
}

llama_status llama_stack_device_status(llama_stack *stk) {
  if (stk == nullptr) return LLAMA_ERR_INVALID_ARG;
  return read_status(stk->status, stk->device, &stk->ws, &stk->dm);
}

size_t llama_kv_cache_bytes(const llama_config *cfg, int32_t max_batch, int32_t max_seq_len) {
  Dims dm;
  if (validate_config(cfg, &dm) != LLAMA_OK || max_batch <= 0 || max_seq_len <= 0) return 0;
  return 2 * (size_t)max_batch * dm.G * (size_t)max_seq_len * dm.D * dm.esize;
}

int32_t llama_ffn_hidden_dim(int32_t d_model, int32_t multiple_of, float ffn_dim_multiplier) {
  if (d_model <= 0 || multiple_of <= 0) return -1;
  long long h = 4LL * d_model;
  h = (2 * h) / 3;
  if (ffn_dim_multiplier > 0.f) h = (long long)((double)ffn_dim_multiplier * (double)h);
  h = (long long)multiple_of * ((h + multiple_of - 1) / multiple_of);
  return h > 0x7fffffffLL ? -1 : (int32_t)h;
}

const char *llama_last_cuda_error(void) { return t_last_cuda_error; }

unsigned long long llama_kernel_launch_count(void) {
  return llama::g_kernel_launches.load(std::memory_order_relaxed);
}

const char *llama_status_string(llama_status s) {
  switch (s) {
    case LLAMA_OK: return "ok";
    case LLAMA_ERR_INVALID_ARG: return "invalid argument";
    case LLAMA_ERR_SHAPE: return "inconsistent shape";
    case LLAMA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LLAMA_ERR_RANGE: return "size or position out of range";
    case LLAMA_ERR_UNSUPPORTED: return "unsupported shape";
    case LLAMA_ERR_OOM: return "device out of memory";
    case LLAMA_ERR_CUDA: return "CUDA error";
    case LLAMA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
