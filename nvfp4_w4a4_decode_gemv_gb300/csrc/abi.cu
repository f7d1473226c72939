// Status strings, argument helpers and the device check of the C ABI.
#include <stdio.h>

#include "common.cuh"

cudaError_t nvfp4_internal_read_error_gemv(unsigned int* out);
cudaError_t nvfp4_internal_read_error_gemv_tc(unsigned int* out);
cudaError_t nvfp4_internal_read_error_reset(unsigned int* out);
cudaError_t nvfp4_internal_read_error_gemm(unsigned int* out);

namespace {
thread_local char g_last_cuda_error[256] = "no CUDA error";
}

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4_OK;
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return NVFP4_ERR_CUDA;
}

bool nvfp4_internal_aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// The library carries sm_103a code only: accept compute capability 10.3.
nvfp4_status nvfp4_internal_check_device() {
  static thread_local int checked_dev = -1;
  static thread_local nvfp4_status verdict = NVFP4_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  if (dev == checked_dev) return verdict;
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  verdict = (major == 10 && minor == 3) ? NVFP4_OK : NVFP4_ERR_DEVICE;
  checked_dev = dev;
  return verdict;
}

extern "C" const char* nvfp4_status_str(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_NULL: return "a required pointer is NULL";
    case NVFP4_ERR_SHAPE: return "a size is out of range or not a required multiple";
    case NVFP4_ERR_ALIGN: return "a pointer is not aligned as required";
    case NVFP4_ERR_RANGE: return "a parameter value is out of range";
    case NVFP4_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case NVFP4_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
  }
  return "unknown status";
}

extern "C" const char* nvfp4_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int nvfp4_version(void) { return (1 << 16) | 0; }

extern "C" nvfp4_status nvfp4_device_status(unsigned int* code) {
  if (!code) return NVFP4_ERR_NULL;
  *code = 0;
  cudaError_t e = nvfp4_internal_read_error_gemv(code);
  if (e == cudaSuccess) e = nvfp4_internal_read_error_gemv_tc(code);
  if (e == cudaSuccess) e = nvfp4_internal_read_error_reset(code);
  if (e == cudaSuccess) e = nvfp4_internal_read_error_gemm(code);
  return nvfp4_internal_cuda_status(e);
}
