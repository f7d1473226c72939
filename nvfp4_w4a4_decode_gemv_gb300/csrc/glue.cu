// Decode-step glue around the NVFP4 projections: the BF16 lm_head GEMV, an
// FP32 -> BF16 cast and an RMS normalization of FP32 rows to BF16.  A Qwen3-style decoder ends in a BF16 lm_head whose logits
// feed the sampler (ReSET reading note §6.4: end-to-end decode on the whole
// model; the lm_head itself is not NVFP4 there).
//
// BF16 GEMV y[m, n] = sum_k x[m, k] w[n, k] (M <= 8): a persistent grid, one
// CTA per SM; each CTA stages x as FP32 in shared memory once, then every warp
// streams groups of 4 weight rows with 128-bit coalesced loads (lanes along K),
// accumulates with packed FP32x2 FMAs and reduces across the warp at the end of
// each row group.  HBM-bound: 2 bytes of weight per 2*M flops.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;                 // weight rows per warp iteration
constexpr int kMaxSmemFloats = 50 * 1024;  // 200 KB of FP32 activations

template <int M>
__global__ void __launch_bounds__(kThreads) bf16_gemv_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ w, int N, int K,
                                                            float* __restrict__ y) {
  extern __shared__ float4 xs4[];
  float* xs = reinterpret_cast<float*>(xs4);
  for (int i = threadIdx.x; i < M * K / 2; i += kThreads) {
    const uint32_t p = __ldg(reinterpret_cast<const uint32_t*>(x) + i);
    xs[2 * i] = bf16_lo(p);
    xs[2 * i + 1] = bf16_hi(p);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (N + kRows - 1) / kRows;
  const int nwarps = gridDim.x * (kThreads / 32);
  for (int g = blockIdx.x * (kThreads / 32) + warp; g < ngroups; g += nwarps) {
    float2 acc[kRows][M];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[r][m] = make_float2(0.f, 0.f);
    const int n0 = g * kRows;
    for (int k = lane * 8; k < K; k += 256) {
      uint4 wv[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int n = n0 + r < N ? n0 + r : N - 1;
        wv[r] = __ldcs(reinterpret_cast<const uint4*>(w + (size_t)n * K + k));
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + m * K + k);
        const float4 xb = *reinterpret_cast<const float4*>(xs + m * K + k + 4);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          acc[r][m] = __ffma2_rn(make_float2(bf16_lo(wv[r].x), bf16_hi(wv[r].x)), make_float2(xa.x, xa.y), acc[r][m]);
          acc[r][m] = __ffma2_rn(make_float2(bf16_lo(wv[r].y), bf16_hi(wv[r].y)), make_float2(xa.z, xa.w), acc[r][m]);
          acc[r][m] = __ffma2_rn(make_float2(bf16_lo(wv[r].z), bf16_hi(wv[r].z)), make_float2(xb.x, xb.y), acc[r][m]);
          acc[r][m] = __ffma2_rn(make_float2(bf16_lo(wv[r].w), bf16_hi(wv[r].w)), make_float2(xb.z, xb.w), acc[r][m]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float s = acc[r][m].x + acc[r][m].y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0 && n0 + r < N) y[(size_t)m * N + n0 + r] = s;
      }
    }
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ x, size_t n8, uint4* __restrict__ y) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = __ldg(x + 2 * i), b = __ldg(x + 2 * i + 1);
    auto pk = [](float lo, float hi) {
      return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
    };
    y[i] = make_uint4(pk(a.x, a.y), pk(a.z, a.w), pk(b.x, b.y), pk(b.z, b.w));
  }
}

// RMS normalization of FP32 rows to BF16, one CTA per row:
//   out[r, k] = BF16( x[r, k] / sqrt( sum_k x[r, k]^2 / K + eps ) )
// Sum of squares in FP32 (per-thread strided partial sums, then a fixed tree
// over the CTA); sqrt and the division are IEEE (sqrtf, __fdiv_rn).
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rms_norm_bf16_kernel(const float* __restrict__ x, int K, long ld,
                                                                     float eps, uint16_t* __restrict__ out) {
  __shared__ float s_warp[kNormThreads / 32];
  __shared__ float s_inv;
  griddep_launch_dependents();
  griddep_wait();             // the input comes from the preceding kernel
  const float* xr = x + (long)blockIdx.x * ld;
  float ss = 0.0f;
  for (int k = threadIdx.x * 4; k < K; k += kNormThreads * 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
    ss = __fmaf_rn(v.x, v.x, ss);
    ss = __fmaf_rn(v.y, v.y, ss);
    ss = __fmaf_rn(v.z, v.z, ss);
    ss = __fmaf_rn(v.w, v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < kNormThreads / 32 ? s_warp[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) s_inv = __fdiv_rn(1.0f, sqrtf(__fadd_rn(__fdiv_rn(t, (float)K), eps)));
  }
  __syncthreads();
  const float inv = s_inv;
  uint16_t* orow = out + (long)blockIdx.x * K;
  for (int k = threadIdx.x * 4; k < K; k += kNormThreads * 4) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v.x, inv))) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v.y, inv))) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v.z, inv))) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v.w, inv))) << 16);
    *reinterpret_cast<uint2*>(orow + k) = make_uint2(lo, hi);
  }
}

template <int M>
cudaError_t launch_bf16(const uint16_t* x, const uint16_t* w, int N, int K, float* y, cudaStream_t stream) {
  static PerDeviceInt sms_cache;   // SM count; the kernel's shared-memory attribute is set per device
  const size_t smem = (size_t)M * K * sizeof(float);
  auto kern = bf16_gemv_kernel<M>;
  cudaError_t err = cudaSuccess;
  const int sms = sms_cache.get([](int dev, cudaError_t* e_out) -> int {
    int n = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bf16_gemv_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemFloats * 4);
    if (e != cudaSuccess) {
      *e_out = e;
      return 0;
    }
    return n > 0 ? n : 1;
  }, &err);
  if (sms == 0) return err;
  kern<<<sms, kThreads, smem, stream>>>(x, w, N, K, y);
  return cudaGetLastError();
}

}  // namespace

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);
nvfp4_status nvfp4_internal_check_device();

extern "C" nvfp4_status nvfp4_bf16_gemv(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                                        cudaStream_t stream) {
  if (!x || !w || !y) return NVFP4_ERR_NULL;
  if (M < 1 || M > 8) return NVFP4_ERR_RANGE;
  if (N < 1 || K < 8 || (K % 8) != 0 || (size_t)M * K > (size_t)kMaxSmemFloats) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(w, 16) || !nvfp4_internal_aligned(y, 16))
    return NVFP4_ERR_ALIGN;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  cudaError_t e;
  switch (M) {
    case 1: e = launch_bf16<1>(x, w, N, K, y, stream); break;
    case 2: e = launch_bf16<2>(x, w, N, K, y, stream); break;
    case 3: e = launch_bf16<3>(x, w, N, K, y, stream); break;
    case 4: e = launch_bf16<4>(x, w, N, K, y, stream); break;
    case 5: e = launch_bf16<5>(x, w, N, K, y, stream); break;
    case 6: e = launch_bf16<6>(x, w, N, K, y, stream); break;
    case 7: e = launch_bf16<7>(x, w, N, K, y, stream); break;
    default: e = launch_bf16<8>(x, w, N, K, y, stream); break;
  }
  return nvfp4_internal_cuda_status(e);
}

extern "C" nvfp4_status nvfp4_f32_to_bf16(const float* x, size_t n, uint16_t* y, cudaStream_t stream) {
  if (n == 0) return NVFP4_OK;
  if (!x || !y) return NVFP4_ERR_NULL;
  if (n % 8) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(y, 16)) return NVFP4_ERR_ALIGN;
  const size_t n8 = n / 8;
  size_t grid = (n8 + 255) / 256;
  if (grid > 4096) grid = 4096;
  f32_to_bf16_kernel<<<(unsigned)grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(x), n8,
                                                         reinterpret_cast<uint4*>(y));
  return nvfp4_internal_cuda_status(cudaGetLastError());
}

extern "C" nvfp4_status nvfp4_rms_norm_bf16(const float* x, int rows, int K, int ld, float eps, uint16_t* out,
                                           cudaStream_t stream) {
  if (rows == 0) return NVFP4_OK;
  if (!x || !out) return NVFP4_ERR_NULL;
  if (rows < 0 || K < 4 || (K % 4) != 0 || ld < K || (ld % 4) != 0) return NVFP4_ERR_SHAPE;
  if (!(eps >= 0.0f)) return NVFP4_ERR_RANGE;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(out, 8)) return NVFP4_ERR_ALIGN;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return nvfp4_internal_cuda_status(cudaLaunchKernelEx(&cfg, rms_norm_bf16_kernel, x, K, (long)ld, eps, out));
}
