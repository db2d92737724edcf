// synth_fill.cu -- device twin of synth/gen.py: fills bf16 tensors with the
// counter-based Irwin-Hall(12) normal variates, bit-identical to the host
// generator, and optionally reduces max |x| (as bf16 bit patterns) for the
// per-tensor scale.  Input generation only: none of the attention or
// quantisation arithmetic lives here.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t normal_bf16_at(uint64_t key, uint64_t idx) {
  int64_t s = 0;
  const uint64_t c0 = idx * 3ull;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t h = mix64(key + (c0 + (uint64_t)j + 1ull) * kGolden);
#pragma unroll
    for (int k = 0; k < 4; ++k) s += (int64_t)((h >> (16 * k)) & 0xFFFFull);
  }
  // (S - 393210) is an integer of magnitude < 2^19: exact in fp32, and the
  // multiplication by 2^-16 is exact as well.
  const float x = __fmul_rn((float)(s - 393210), 1.0f / 65536.0f);
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__global__ void normal_bf16_kernel(uint16_t* __restrict__ out, uint64_t key, uint64_t base,
                                   int64_t n, unsigned int* __restrict__ amax_bits) {
  unsigned int local = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint16_t b = normal_bf16_at(key, base + (uint64_t)i);
    if (out) out[i] = b;
    const unsigned int mag = b & 0x7FFFu;
    local = mag > local ? mag : local;
  }
  if (amax_bits) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned int other = __shfl_xor_sync(0xFFFFFFFFu, local, o);
      local = other > local ? other : local;
    }
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, local);
  }
}

}  // namespace

extern "C" {

// out: device bf16 buffer of n elements, or NULL to only reduce.
// amax_bits: device uint32 that receives max over elements of (bf16 bits & 0x7FFF)
// (atomicMax, caller initialises), or NULL.
int synth_normal_bf16(void* out, uint64_t key, uint64_t base, int64_t n, unsigned int* amax_bits,
                      cudaStream_t stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 132) * 16;
  if (blocks > cap) blocks = cap;
  normal_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>((uint16_t*)out, key, base, n, amax_bits);
  return (int)cudaGetLastError();
}

}  // extern "C"
