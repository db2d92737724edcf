// pfkv_internal.h -- host-side helpers shared by the libpfkv translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "pfkv.h"

namespace pfkv {

// Records a printf-style message for pfkv_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Clears the calling thread's last-error message.
void clear_error();
// Returns PFKV_OK or PFKV_ERR_CUDA (with a message) after a launch sequence.
int check_cuda(const char* what);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Number of SMs of the current device (queried each call; cheap).
int device_sm_count();

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute belongs to each device's context);
// `done` is the call site's mask of devices (0-63) already set.
int set_max_dynamic_smem(const void* func, int bytes, std::atomic<uint64_t>& done, const char* what);

// Encodes a tiled TMA descriptor through the driver entry point obtained from
// the runtime (no link-time dependency on libcuda).
int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                      const cuuint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace pfkv
