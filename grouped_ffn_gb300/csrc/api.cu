// Library-wide C entry points: workspace set-up, device status read-back,
// status strings, and the per-device SM-count cache.
#include <mutex>

#include "common.cuh"

namespace moe_host {

int sm_count() {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < kMaxDevices) cache[dev] = n;
  return n;
}

}  // namespace moe_host

extern "C" moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (moe_status s = moe_host::check_ws(ws, ws_bytes, moe::kStatusBytes)) return s;
  return cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

extern "C" moe_status moe_check_device_status(void *ws, void *stream, int32_t *info_host) {
  if (moe_status s = moe_host::check_ws(ws, moe::kStatusBytes, moe::kStatusBytes)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t words[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(words, ws, sizeof(words), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (words[0] != 0) {
    if (cudaMemsetAsync(ws, 0, 3 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (info_host) *info_host = words[1];
  return static_cast<moe_status>(words[0]);
}

extern "C" const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_INDEX: return "device: index out of range";
    case MOE_ERR_DEVICE_TIMEOUT: return "device: bounded wait expired";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_PLACEMENT: return "device: placement tables inconsistent";
  }
  return "unknown status";
}

extern "C" const char *moe_version(void) { return "grouped_ffn_gb300 0.1 (sm_103a)"; }
