// Test-only helper: the GPU's own fp32 -> e4m3 conversion
// (cvt.rn.satfinite.e4m3x2.f32: round to nearest even, finite overflow and
// infinities clamped to +-448) over a range of fp32 bit patterns, so that the
// oracle's encoder can be compared with the hardware routine on every fp32
// value.  Not part of the library.
#include <cstdint>
#include <cuda_runtime.h>

__global__ void e4m3_cvt_range_kernel(uint32_t start, uint8_t* out, uint32_t n) {
  const uint32_t i = 2u * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float lo = __uint_as_float(start + i), hi = __uint_as_float(start + i + 1u);
  uint16_t r;
  // the first source operand fills the upper byte, the second the lower one
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tmov.b16 %0, t;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
  out[i] = (uint8_t)(r & 0xFFu);
  out[i + 1u] = (uint8_t)(r >> 8);
}

// Codes of the fp32 values with bit patterns start .. start + n - 1 into the
// device buffer out[n] (n even, start + n <= 2^32), on the legacy default
// stream.  Returns the CUDA error code of the launch.
extern "C" __attribute__((visibility("default"))) int e4m3_cvt_range(uint32_t start, void* out, uint32_t n) {
  if (n == 0u) return 0;
  if (n & 1u) return (int)cudaErrorInvalidValue;
  const uint32_t threads = 256u, pairs = n / 2u;
  e4m3_cvt_range_kernel<<<(pairs + threads - 1u) / threads, threads>>>(start, static_cast<uint8_t*>(out), n);
  return (int)cudaGetLastError();
}
