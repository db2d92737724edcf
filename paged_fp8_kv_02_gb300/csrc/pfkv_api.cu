// pfkv_api.cu -- error reporting, device queries, TMA descriptor encoding and
// the small status/version entry points of libpfkv.
#include <cudaTypedefs.h>
#include <string.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {

namespace {
thread_local char g_msg[512] = "";
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_msg[0] = '\0'; }

int check_cuda(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PFKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return PFKV_OK;
}

int set_max_dynamic_smem(const void* func, int bytes, std::atomic<uint64_t>& done, const char* what) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_cuda(what);
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return PFKV_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return check_cuda(what);
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return PFKV_OK;
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                      const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
      return fail(PFKV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint32_t estrides[5] = {1, 1, 1, 1, 1};
  CUresult r = encode(map, dtype, rank, base, dims, strides_bytes, box, estrides,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PFKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PFKV_OK;
}

namespace {
// One thread waits, through the same bounded wait the kernels use, on an
// mbarrier that nothing ever arrives on; the wait gives up after about one
// second and the kernel reports the timeout bit.
__global__ void barrier_timeout_selftest_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  *status = mbar_wait(b, 0) ? 0 : kErrWaitTimeout;
}
}  // namespace

}  // namespace pfkv

extern "C" {

int pfkv_selftest_barrier_timeout(int32_t* d_status, pfkv_stream_t stream) {
  pfkv::clear_error();
  if (d_status == nullptr) return pfkv::fail(PFKV_ERR_INVALID_ARG, "selftest: null status pointer");
  pfkv::barrier_timeout_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d_status);
  return pfkv::check_cuda("selftest launch");
}

const char* pfkv_last_error(void) { return pfkv::g_msg; }

const char* pfkv_version(void) { return "pfkv 0.1 (sm_103a)"; }

int pfkv_workspace_status(const void* workspace, int32_t* status, pfkv_stream_t stream) {
  pfkv::clear_error();
  if (workspace == nullptr || status == nullptr)
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "workspace_status: null pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return pfkv::check_cuda("workspace_status memcpy");
  if (cudaStreamSynchronize(s) != cudaSuccess) return pfkv::check_cuda("workspace_status sync");
  return PFKV_OK;
}

}  // extern "C"
