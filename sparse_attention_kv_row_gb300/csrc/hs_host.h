// hs_host.h -- host-side helpers shared by the library's translation units:
// per-thread error message, device properties cache, pointer classification.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/hisparse.h"

namespace hs {

// Records `msg` as the calling thread's last error and returns `code`.
hs_err fail(hs_err code, const char* fmt, ...);
void clear_error();

struct DeviceInfo {
  int device;
  int sm_count;
  int max_smem_optin;
  int max_smem_per_sm;
};
// Properties of the current device (cached per device).
hs_err current_device(DeviceInfo* out);

enum class MemKind { kDevice, kHost, kManaged, kUnregistered, kUnknown };
MemKind classify(const void* p);

// A named NVTX range around one C-ABI call when the environment variable
// HS_NVTX is set to anything but "0" (read once per process); otherwise it
// does nothing.  For timelines taken with a profiler.
class CallRange {
 public:
  explicit CallRange(const char* name);
  ~CallRange();
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;

 private:
  bool on_;
};

// Lemire-Kaser-Kurz divider constant for 1 <= d < 2^32 (d == 1 gives magic 0
// and the device side short-circuits it).
inline uint64_t fastdiv_magic(uint32_t d) { return d <= 1 ? 0ull : (~0ull) / d + 1ull; }

}  // namespace hs
