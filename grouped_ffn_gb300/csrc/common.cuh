// Shared helpers of the MoE hot-path library (device status word, bounded
// waits, argument checks).  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Kernel ids recorded with a device error (status word [2]).
enum KernelId : int32_t {
  K_ROUTE = 1,
  K_LAYOUT_SCAN = 2,
  K_LAYOUT_FINALIZE = 3,
  K_PERMUTE = 4,
  K_FFN_GATE_UP = 5,
  K_FFN_DOWN = 6,
  K_COMBINE = 7,
  K_BALANCE = 8,
  K_SELFTEST = 9,
};

// Status block at the start of every workspace (int32 words):
//   [0] first device error code (moe_status), 0 = none
//   [1] detail (offending index, or elapsed wait in microseconds)
//   [2] KernelId of the reporter
constexpr size_t kStatusBytes = MOE_WS_STATUS_BYTES;
// Status-block word [16]: the grouped FFN's count of finished CTAs; the
// last CTA of a launch clears it and the per-segment readiness counters.
constexpr int kFfnExitWord = 16;

// Workspace map (bytes): [0, 256) status block; [256, 256 + 4 * 1024) the
// grouped FFN's per-segment readiness counters; [4352, 4608) the layout's
// tile ticket; [4608, ...) the layout's look-back flags.
constexpr size_t kFfnReadyOff = kStatusBytes;
constexpr size_t kLayoutTicketOff = kFfnReadyOff + 4 * 1024;
constexpr size_t kLayoutFlagsOff = kLayoutTicketOff + 256;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void report_error(int32_t *status, int32_t code, int32_t info,
                                             int32_t kernel) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) {
    atomicExch(status + 1, info);
    atomicExch(status + 2, kernel);
  }
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_stream_u4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Programmatic dependent launch: wait until the grids this one depends on
// have finished and their writes are visible (a no-op when the kernel was
// launched without the attribute), and let the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace moe

// ---------------------------------------------------------------- host side
namespace moe_host {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int32_t *status_ptr(void *ws) { return reinterpret_cast<int32_t *>(ws); }

// Number of SMs of the current device (cached per device id).
int sm_count();

// Maps the last CUDA launch error to a status.
inline moe_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Launch with programmatic stream serialization: the kernel may begin while
// its predecessor on the stream drains; it calls moe::pdl_wait() before
// touching anything the predecessor writes.
template <typename... KArgs, typename... Args>
inline moe_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Cooperative launch (every CTA resident at once, so CTAs may wait for one
// another) with programmatic stream serialization as well.
template <typename... KArgs, typename... Args>
inline moe_status launch_coop_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline moe_status check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || !aligned16(ws) || ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

}  // namespace moe_host
