// Shared device helpers for the decoder-block kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

namespace llama {

typedef __nv_bfloat16 bf16;

// Each block / stack handle owns one device status word (an int in device
// memory).  A kernel whose bounded wait runs out, or that meets an invalid
// token id, records the first such event there instead of trapping; the host
// reads and clears it with llama_block_device_status().
enum DeviceStatusCode : int {
  DEV_OK = 0,
  DEV_TIMEOUT_PRODUCER = 1,
  DEV_TIMEOUT_MMA = 2,
  DEV_TIMEOUT_EPILOGUE = 3,
  DEV_TIMEOUT_ATTN = 4,
  DEV_TIMEOUT_PHASE = 5,  // fused decode kernel: a phase barrier wait ran out
  DEV_BAD_TOKEN = 16,
};

// Remembers the last CUDA error of a failing library call in this host thread
// (read through llama_last_cuda_error()).
void note_cuda_error(cudaError_t e);
// Counts one kernel launch (library-wide total, read by llama_kernel_launch_count).
void count_launch();
// Identifier of the CUDA context current on the calling thread, unique within
// the process (a context created after a device reset gets a new one); 0 when
// no context is current or the driver cannot tell.
unsigned long long current_context_id();

// Runs a per-context set-up (a kernel's shared-memory limit, a symbol's device
// address) once in every CUDA context it is needed in: each device has its own
// context, and a device reset replaces it.  Until the set-up has succeeded in
// the current context it is run again on the next call.
class PerContextOnce {
 public:
  template <typename F> cudaError_t run(F &&init) {
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mutex_);
    if (id != 0)
      for (unsigned long long done : done_)
        if (done == id) return cudaSuccess;
    const cudaError_t e = init();
    if (e == cudaSuccess && id != 0) done_.push_back(id);
    return e;
  }

 private:
  std::mutex mutex_;
  std::vector<unsigned long long> done_;
};

__device__ __forceinline__ void report_status(int *status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  uint4 raw;
  __device__ __forceinline__ float get(int i) const {
    const T *p = reinterpret_cast<const T *>(&raw);
    return to_f32<T>(p[i]);
  }
  __device__ __forceinline__ void set(int i, float v) {
    T *p = reinterpret_cast<T *>(&raw);
    p[i] = from_f32<T>(v);
  }
};

template <typename T> __device__ __forceinline__ Vec16<T> load16(const T *p) {
  Vec16<T> v;
  v.raw = *reinterpret_cast<const uint4 *>(p);
  return v;
}
template <typename T> __device__ __forceinline__ void store16(T *p, const Vec16<T> &v) {
  *reinterpret_cast<uint4 *>(p) = v.raw;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// SiLU(z) = z * sigmoid(z) = z / (1 + e^-z).  The quotient uses the fast
// division intrinsic (about 2 ulp; z -> -inf gives -0, z -> +inf gives z):
// the IEEE-exact division is a long dependent sequence that dominated the
// SwiGLU epilogue when only a few warps per SM are live (decode shapes).
__device__ __forceinline__ float silu_f32(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Programmatic dependent launch.  A kernel started with launch_pdl may begin
// while the previous kernel on the stream is still running: before it reads
// anything an earlier kernel wrote, or writes anything, it calls
// grid_dependency_wait(), which returns once every earlier kernel of the stream
// has completed and its memory is visible (at once when there is none).  Work
// that touches only data no kernel writes -- the weights -- may come first.
// allow_dependents_launch() lets the next such kernel be scheduled early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Budget for a bounded spin on an mbarrier or flag, in SM clock cycles
// (about 2 s at 2 GHz); long enough that no legitimate wait reaches it.
constexpr long long kWaitBudgetCycles = 4000000000LL;

// A handle's device status block.  The `int *status` the kernels receive
// points at `code` (or is null).  `wait_budget` is set from the host
// (llama_block_set_wait_budget / llama_stack_set_wait_budget): it bounds, in
// SM clock cycles, every wait that gives up (0 means kWaitBudgetCycles).
// Waits that drain copies and MMAs already in flight before a CTA reuses their
// memory or exits (ptx::mbar_drain) always use kWaitBudgetCycles.
struct DeviceStatus {
  int code;
  int reserved;
  long long wait_budget;
};

__device__ __forceinline__ long long wait_budget(const int *status) {
  if (status == nullptr) return kWaitBudgetCycles;
  const long long b = __ldg(&reinterpret_cast<const DeviceStatus *>(status)->wait_budget);
  return b > 0 ? b : kWaitBudgetCycles;
}

}  // namespace llama
