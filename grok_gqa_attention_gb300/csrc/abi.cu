// Host-side helpers of the C ABI: error text, device checks, tensor maps.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "host.cuh"

namespace grok {

static thread_local char g_error[512] = "";

grok_status fail(grok_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_error, sizeof(g_error), fmt, ap);
  va_end(ap);
  return s;
}

grok_status cuda_status(cudaError_t e) {
  switch (e) {
    case cudaSuccess:
      return GROK_OK;
    case cudaErrorECCUncorrectable:
    case cudaErrorNvlinkUncorrectable:
    case cudaErrorContained:
    case cudaErrorIllegalAddress:
    case cudaErrorLaunchTimeout:
    case cudaErrorAssert:
    case cudaErrorHardwareStackError:
    case cudaErrorIllegalInstruction:
    case cudaErrorMisalignedAddress:
    case cudaErrorInvalidAddressSpace:
    case cudaErrorInvalidPc:
    case cudaErrorLaunchFailure:
    case cudaErrorTensorMemoryLeak:
    case cudaErrorExternalDevice:
      return GROK_ERR_DEVICE_FAULT;
    default:
      return GROK_ERR_CUDA;
  }
}

grok_status device_index(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(cuda_status(e), "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fail(GROK_ERR_UNSUPPORTED, "device index %d out of range", *dev);
  return GROK_OK;
}

grok_status device_sm_count(int* sm_count) {
  static int cache[kMaxDevices] = {0};  // 0 = unknown, -1 = unsupported, else SM count
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(cuda_status(e), "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) {
    *sm_count = cache[dev];
    return GROK_OK;
  }
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return fail(cuda_status(e), "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(GROK_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                major, minor);
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = sms;
  *sm_count = sms;
  return GROK_OK;
}

grok_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(cuda_status(e), "%s launch: %s", what, cudaGetErrorString(e));
  return GROK_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static grok_status encode_tmap_16bit_4d(CUtensorMapDataType type, CUtensorMap* map, const void* base,
                                       const uint64_t dims[4], const uint64_t strides[3], const uint32_t box[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(GROK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gstr[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, type, 4, const_cast<void*>(base), gdim, gstr, bdim, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GROK_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
  return GROK_OK;
}

grok_status encode_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                                const uint64_t strides[3], const uint32_t box[4]) {
  return encode_tmap_16bit_4d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, dims, strides, box);
}

grok_status encode_tmap_f16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                               const uint64_t strides[3], const uint32_t box[4]) {
  return encode_tmap_16bit_4d(CU_TENSOR_MAP_DATA_TYPE_FLOAT16, map, base, dims, strides, box);
}

grok_status encode_tmap_u8_2d(CUtensorMap* map, const void* base, const uint64_t dims[2], uint64_t row_stride,
                              const uint32_t box[2]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(GROK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[2] = {dims[0], dims[1]};
  cuuint64_t gstr[1] = {row_stride};
  cuuint32_t bdim[2] = {box[0], box[1]};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstr, bdim, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GROK_ERR_CUDA, "cuTensorMapEncodeTiled (uint8) failed (CUresult %d)", int(r));
  return GROK_OK;
}

}  // namespace grok

extern "C" int grok_abi_version(void) { return GROK_ATTN_ABI_VERSION; }

extern "C" const char* grok_last_error(void) { return grok::g_error; }

extern "C" grok_status grok_cuda_error_status(int cuda_error) {
  return grok::cuda_status(static_cast<cudaError_t>(cuda_error));
}
