// Library-wide entry points: status strings, ABI version, device check and
// the device error word.
#include <atomic>

#include <cuda_runtime.h>

#include "common.cuh"
#include "host_common.h"
#include "specv.h"

namespace specv {

namespace {
constexpr int kMaxDevices = 64;
// 0 = unknown, 1 = supported, 2 = unsupported
std::atomic<int> g_device_ok[kMaxDevices];
}  // namespace

specv_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPECV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPECV_ERR_UNSUPPORTED;
  int state = g_device_ok[dev].load(std::memory_order_relaxed);
  if (state == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SPECV_ERR_CUDA;
    state = (major == 10 && minor == 3) ? 1 : 2;
    g_device_ok[dev].store(state, std::memory_order_relaxed);
  }
  return state == 1 ? SPECV_OK : SPECV_ERR_UNSUPPORTED;
}

}  // namespace specv

extern "C" const char* specv_status_string(specv_status status) {
  switch (status) {
    case SPECV_OK: return "ok";
    case SPECV_ERR_INVALID_ARG: return "invalid argument";
    case SPECV_ERR_UNSUPPORTED: return "unsupported device or shape";
    case SPECV_ERR_CUDA: return "CUDA error";
    case SPECV_ERR_DEVICE_DATA: return "device-detected invalid data";
    case SPECV_ERR_TIMEOUT: return "bounded device wait expired";
    case SPECV_ERR_SCRATCH_LIMIT: return "shape exceeds the built-in scratch of the allocation-free call";
  }
  return "unknown status";
}

extern "C" int specv_abi_version(void) { return SPECV_ABI_VERSION; }

extern "C" specv_status specv_read_device_error(const void* workspace, void* stream, int32_t* status_out) {
  if (!workspace || !status_out || !specv::aligned_to(workspace, 256)) return SPECV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPECV_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SPECV_ERR_CUDA;
  *status_out = v;
  return SPECV_OK;
}

namespace {

// One thread waits on a barrier that nothing arrives at (unless `arrive`),
// with the poll-limited wait of the production kernels.
__global__ void bounded_wait_kernel(uint32_t max_polls, int arrive, void* workspace) {
  __shared__ uint64_t bar;
  specv::mbar_init(&bar, 1);
  specv::fence_mbar_init();
  if (arrive) specv::mbar_arrive(&bar);
  const bool ok = specv::mbar_wait_parity(&bar, 0, max_polls);
  *reinterpret_cast<int*>(workspace) = ok ? SPECV_OK : SPECV_ERR_TIMEOUT;
}

}  // namespace

extern "C" specv_status specv_selftest_bounded_wait(uint32_t max_polls, int arrive, void* workspace,
                                                   size_t workspace_bytes, void* stream) {
  if (max_polls < 1 || max_polls > 65536 || !workspace || workspace_bytes < 256 ||
      !specv::aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  const specv_status s = specv::check_device();
  if (s != SPECV_OK) return s;
  bounded_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(max_polls, arrive, workspace);
  return cudaGetLastError() == cudaSuccess ? SPECV_OK : SPECV_ERR_CUDA;
}
