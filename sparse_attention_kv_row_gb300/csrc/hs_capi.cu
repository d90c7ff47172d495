// hs_capi.cu -- error reporting, device-property cache, pointer classification
// and the small informational entry points of the C ABI.
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "hs_host.h"

namespace hs {

namespace {
thread_local char g_last_error[512] = {0};

std::mutex g_dev_mu;
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {false};
}  // namespace

hs_err fail(hs_err code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_last_error[0] = 0; }

hs_err current_device(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(HS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(HS_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev_ok[dev]) {
    DeviceInfo d{dev, 0, 0, 0};
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&d.max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                 dev);
    if (e != cudaSuccess)
      return fail(HS_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    g_dev[dev] = d;
    g_dev_ok[dev] = true;
  }
  *out = g_dev[dev];
  return HS_OK;
}

namespace {
bool nvtx_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("HS_NVTX");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}
}  // namespace

CallRange::CallRange(const char* name) : on_(nvtx_enabled()) {
  if (on_) nvtxRangePushA(name);
}
CallRange::~CallRange() {
  if (on_) nvtxRangePop();
}

MemKind classify(const void* p) {
  cudaPointerAttributes attr{};
  const cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return MemKind::kUnknown;
  }
  switch (attr.type) {
    case cudaMemoryTypeDevice: return MemKind::kDevice;
    case cudaMemoryTypeHost: return MemKind::kHost;
    case cudaMemoryTypeManaged: return MemKind::kManaged;
    default: return MemKind::kUnregistered;
  }
}

}  // namespace hs

extern "C" const char* hs_err_string(int32_t err) {
  switch (err) {
    case HS_OK: return "HS_OK";
    case HS_ERR_ARG: return "HS_ERR_ARG: invalid argument";
    case HS_ERR_UNSUPPORTED: return "HS_ERR_UNSUPPORTED: outside the supported limits";
    case HS_ERR_CUDA: return "HS_ERR_CUDA: CUDA runtime or launch error";
    default: return "unknown hs_err";
  }
}

extern "C" const char* hs_status_string(int32_t bit) {
  switch (bit) {
    case HS_ST_DUP_ID: return "HS_ST_DUP_ID";
    case HS_ST_BAD_POOL_ROW: return "HS_ST_BAD_POOL_ROW";
    case HS_ST_BAD_LRU_SLOT: return "HS_ST_BAD_LRU_SLOT";
    case HS_ST_BAD_HOT_ROW: return "HS_ST_BAD_HOT_ROW";
    case HS_ST_TIMEOUT: return "HS_ST_TIMEOUT";
    case HS_ST_BAD_STATE: return "HS_ST_BAD_STATE";
    case HS_ST_BAD_INDEX: return "HS_ST_BAD_INDEX";
    default: return "";
  }
}

extern "C" const char* hs_last_error(void) { return hs::g_last_error; }

extern "C" int32_t hs_abi_version(void) { return HS_ABI_VERSION; }
