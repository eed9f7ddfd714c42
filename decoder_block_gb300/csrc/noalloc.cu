// Decode-step attention that allocates nothing (llama_op_attention_decode_noalloc).
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code that executes while another component owns every device allocation
// (a serving engine's pre-reserved memory pool, an embedded runtime with a
// fixed memory budget, or a host thread that must not synchronise the device
// the way an allocation can).  For them this entry point keeps the split-KV
// partials of the decode kernel in one file-scope device array that the
// library image carries, instead of caller- or library-allocated memory.
//
// The array is part of the loaded library on every GPU that uses it and stays
// resident until the process exits.  Its device address is looked up once per
// CUDA context -- on the first call made with a device current, and again
// after that device's context was reset -- so make the first call on each
// device before any stream capture.  All calls share the one array, so calls
// whose kernels could run at the same time on the GPU (different streams
// without ordering between them) race on it.
#include <mutex>

#include "llama_ops.h"
#include "kernels.h"
#include "tc_kernels.h"

using namespace llama;

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[LLAMA_NOALLOC_SCRATCH_BYTES];

// The array's device address in each CUDA context that has used it.  A
// device reset ends the context and unloads the library image from it; the
// context created after it has another identifier, so the address is looked
// up again instead of reusing a stale one.
struct ScratchAddress {
  unsigned long long context;
  void *ptr;
};
constexpr int kMaxContexts = 64;
std::mutex g_setup_mutex;
ScratchAddress g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

// Device address of g_decode_scratch in the current context (set-up on first use).
llama_status scratch_address(void **out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  unsigned long long ctx = current_context_id();
  if (ctx != 0)
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch[i].context == ctx) {
        *out = g_scratch[i].ptr;
        return LLAMA_OK;
      }
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return LLAMA_ERR_CUDA;
  }
  ctx = current_context_id();  // the look-up makes a context current if none was
  if (ctx != 0) {
    if (g_scratch_n == kMaxContexts) g_scratch_n = 0;  // many resets: start the table over
    g_scratch[g_scratch_n++] = ScratchAddress{ctx, p};
  }
  *out = p;
  return LLAMA_OK;
}

llama_status check_ptr(const void *p) {
  if (p == nullptr) return LLAMA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return LLAMA_ERR_ALIGN;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return LLAMA_ERR_INVALID_ARG;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) ? LLAMA_OK : LLAMA_ERR_INVALID_ARG;
}

}  // namespace

extern "C" llama_status llama_op_attention_decode_noalloc(const void *q, const llama_kv_cache *kv, void *o,
                                                          int32_t B, int32_t start_pos, int32_t H, int32_t G,
                                                          int32_t D, llama_stream stream) {
  if (kv == nullptr || B <= 0 || start_pos < 0 || H <= 0 || G <= 0 || D <= 0) return LLAMA_ERR_INVALID_ARG;
  if (H % G != 0) return LLAMA_ERR_SHAPE;
  if (!attn_decode_supported(H, G, D)) return LLAMA_ERR_UNSUPPORTED;
  if (B > kv->max_batch || (long long)start_pos + 1 > kv->max_seq_len) return LLAMA_ERR_RANGE;
  // Partials: H x ceil((start_pos + 1) / 256) chunks x (D + 2) floats per sequence; with a single chunk the
  // kernel writes o directly and uses none.  Batches whose partials exceed the array run in groups of
  // sequences, one group after another on the stream, each reusing it: one sequence's partials must fit.
  const size_t n_split = (size_t)((start_pos + 1 + 255) / 256);
  const size_t per_seq = n_split > 1 ? (size_t)H * n_split * (D + 2) * sizeof(float) : 0;
  if (per_seq > (size_t)LLAMA_NOALLOC_SCRATCH_BYTES) return LLAMA_ERR_RANGE;
  for (const void *p : {q, (const void *)kv->k, (const void *)kv->v, (const void *)o}) {
    llama_status c = check_ptr(p);
    if (c != LLAMA_OK) return c;
  }
  void *scratch = nullptr;
  llama_status s = scratch_address(&scratch);
  if (s != LLAMA_OK) return s;
  // Every partial slot the combine step reads is written by the same call
  // first, so nothing in the array has to be cleared between calls.
  AttnScratch ws;
  ws.partial = scratch;
  ws.bytes = LLAMA_NOALLOC_SCRATCH_BYTES;
  cudaError_t e = launch_attn_decode((const bf16 *)q, (const bf16 *)kv->k, (const bf16 *)kv->v, (bf16 *)o, B,
                                     start_pos, H, G, D, kv->max_seq_len, ws, nullptr, (cudaStream_t)stream);
  return e == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA;
}
