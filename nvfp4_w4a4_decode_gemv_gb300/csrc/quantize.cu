// BF16 -> NVFP4 quantizer (E2M1 codes, E4M3 block scales, FP32 global scale).
//
// Format: ReSET reading note §2.1 and §6.1 (E2M1 elements, E4M3 scale per
// 16-element block, FP32 global scale); the activation quantizer "Q" feeding
// the GEMV with a non-interleaved scale layout: reading note §5.3 (Table 3).
//
// The recipe is evaluated with one IEEE rounding per operation (__fdiv_rn,
// __fmul_rn: no contraction, no approximate reciprocal), so codes and scales
// are bit-identical to a plain FP32 evaluation of the recipe:
//   g = amax / 2688;  s = E4M3(bm / (6 g));  code = E2M1(x / (dec(s) g)).
// The element codes come from x times the IEEE reciprocal of the scale where
// that provably gives the quotient's code (see quant_block), else from the
// IEEE quotient itself.
//
// Two launch shapes:
//  * activations (up to 8 blocks of 16 per thread of one cluster of up to 16
//    CTAs x 512 threads): ONE launch of a thread-block cluster; every CTA
//    keeps its blocks in registers, the tensor amax is reduced across the
//    cluster through distributed shared memory, then codes are written
//    without a second read of x.  rms_norm_quant_kernel is the same pattern
//    with the decode step's RMS normalization in front (one CTA per row).
//  * larger tensors (offline weight quantization): amax kernel (atomicMax on
//    the float bits, which order like the values for non-negative floats, into
//    the global-scale slot), a grid-stride quantize kernel that reads that amax,
//    and a one-thread kernel that turns amax into amax / 2688.
#include <stdlib.h>

#include "common.cuh"
#include "quant_block.cuh"

namespace {

constexpr int kThreads = 256;          // multi-launch (weight-sized) path
constexpr int kCThreads = 512;         // single-launch cluster path
constexpr int kMaxCluster = 16;        // non-portable cluster size, capped by the device
constexpr float kGlobalDivisor = 2688.0f;   // 448 * 6

// ---- element sources: block b of a [rows, K] tensor -> 16 floats ----------
// Each source returns values that are exactly representable in BF16.
// Loads are L2-only (ld.global.cg): the kernels ask L2 for their input before
// waiting on the preceding kernel, which may still be writing it, and a
// non-coherent load after the wait was measured to return pre-wait data in
// that case; L2 is coherent.
struct SrcBF16 {
  const uint16_t* x;
  int nbr;      // blocks per row = K / 16
  int K;
  __device__ void prefetch(long b) const { prefetch_l2(x + (b / nbr) * (long)K + (b % nbr) * 16); }
  __device__ void load(long b, float v[16]) const {
    const long r = b / nbr, c = b % nbr;
    const uint4* p = reinterpret_cast<const uint4*>(x + r * (long)K + c * 16);
    const uint4 a = __ldcg(p), d = __ldcg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, d.x, d.y, d.z, d.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(w[i]);
      v[2 * i + 1] = bf16_hi(w[i]);
    }
  }
};

NVFP4_DEVINL float round_bf16(float f) {
  return __bfloat162float(__float2bfloat16_rn(f));
}

struct SrcF32 {
  const float* x;
  int nbr;
  long ld;
  __device__ void prefetch(long b) const { prefetch_l2(x + (b / nbr) * ld + (b % nbr) * 16); }
  __device__ void load(long b, float v[16]) const {
    const long r = b / nbr, c = b % nbr;
    const float4* p = reinterpret_cast<const float4*>(x + r * ld + c * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = __ldcg(p + i);
      v[4 * i] = round_bf16(q.x);
      v[4 * i + 1] = round_bf16(q.y);
      v[4 * i + 2] = round_bf16(q.z);
      v[4 * i + 3] = round_bf16(q.w);
    }
  }
};

// SiLU(gate) * up, FP32, rounded to BF16.  gate = columns [0, I), up = [I, 2I).
struct SrcSiluMul {
  const float* gu;
  int nbr;   // I / 16
  int I;
  __device__ void prefetch(long b) const {
    const float* pg = gu + (b / nbr) * 2L * I + (b % nbr) * 16;
    prefetch_l2(pg);
    prefetch_l2(pg + I);
  }
  __device__ void load(long b, float v[16]) const {
    const long r = b / nbr, c = b % nbr;
    const float4* pg = reinterpret_cast<const float4*>(gu + r * 2L * I + c * 16);
    const float4* pu = reinterpret_cast<const float4*>(gu + r * 2L * I + I + c * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 g = __ldcg(pg + i), u = __ldcg(pu + i);
      const float gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float s = __fdiv_rn(gs[j], __fadd_rn(1.0f, expf(-gs[j])));
        v[4 * i + j] = round_bf16(__fmul_rn(s, us[j]));
      }
    }
  }
};

// ---- single-launch cluster path --------------------------------------------
template <class Src, int NB>
__global__ void __launch_bounds__(kCThreads) quant_cluster_kernel(Src src, long nblocks, uint8_t* codes,
                                                                  uint8_t* scales, float* global, int trigger_late) {
  __shared__ float s_warp[kCThreads / 32];
  __shared__ float s_peer[kMaxCluster];      // slot r: the maximum of CTA r of the cluster
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = gridDim.x;          // the whole grid is one cluster
  // Peers may write into this CTA's shared memory only once it runs: arrive
  // now, wait just before the first remote store.
  if (csize > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // Programmatic dependent launch: let the next kernel (the GEMV) start
  // launching at once -- it reads only weights until it waits on this grid, so
  // its CTAs take over SMs as the preceding GEMV's CTAs leave and prefetch their
  // first weight tiles -- then wait for the preceding kernel, which may produce
  // this kernel's input.
  // Before that wait, ask L2 for this thread's input: when the input does not
  // come from the preceding kernel, its HBM latency overlaps that kernel's
  // tail; when it does, the hint is harmless (the loads below come after the
  // wait and see the preceding kernel's writes).
  if (!trigger_late) griddep_launch_dependents();
  const long T = (long)csize * kCThreads;
  const long gt = (long)rank * kCThreads + threadIdx.x;
#pragma unroll
  for (int i = 0; i < NB; ++i)
    if (gt + i * T < nblocks) src.prefetch(gt + i * T);
  griddep_wait();

  float v[NB][16];
  float bm[NB];
  float local = 0.0f;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const long b = gt + i * T;
    if (b < nblocks) {
      src.load(b, v[i]);
      bm[i] = block_absmax(v[i]);
      local = fmaxf(local, bm[i]);
    } else {
      bm[i] = 0.0f;
    }
  }
  if (trigger_late) griddep_launch_dependents();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local = fmaxf(local, __shfl_xor_sync(0xffffffffu, local, o));
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = local;
  __syncthreads();
  // Every warp reduces the warp maxima itself: no second block barrier.
  const int lane = threadIdx.x & 31;
  float amax = lane < kCThreads / 32 ? s_warp[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (csize > 1) {
    // Push this CTA's maximum into slot `rank` of every CTA, then one cluster
    // barrier (release / acquire); after it each CTA reads only its own shared
    // memory, so no CTA touches a peer's once the barrier has passed.
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (threadIdx.x < csize) st_dsmem_f32(dsmem_addr(&s_peer[rank], threadIdx.x), amax);
    cluster_sync();
    amax = lane < (int)csize ? s_peer[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  const float g = __fdiv_rn(amax, kGlobalDivisor);
  if (rank == 0 && threadIdx.x == 0) *global = g;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const long b = gt + i * T;
    if (b < nblocks) {
      uint2 c;
      const uint32_t s = quant_block(v[i], bm[i], g, c);
      reinterpret_cast<uint2*>(codes)[b] = c;
      scales[b] = static_cast<uint8_t>(s);
    }
  }
}

// ---- RMS normalization fused with the quantizer ----------------------------
// One CTA per row, the call's rows forming one cluster.  Thread t of CTA r owns
// block t of row r (16 FP32 values, kept in registers from the load to the
// codes).  The row's sum of squares is reduced in the CTA (each thread's 16
// squares in order, then a fixed shuffle tree), the normalized values are
// rounded to BF16 exactly as nvfp4_rms_norm_bf16 rounds them
// (BF16(x * (1 / sqrt(ss / K + eps))), IEEE division and square root), and
// the tensor amax of those BF16 values goes through the cluster as in
// quant_cluster_kernel.  The BF16 row can be written out as well.
constexpr int kMaxNormQRows = 8;           // cluster size: portable
constexpr int kMaxNormQThreads = 1024;     // K / 16 <= 1024

__global__ void __launch_bounds__(kMaxNormQThreads) rms_norm_quant_kernel(const float* __restrict__ x, int K, long ld,
                                                                          float eps, uint8_t* codes, uint8_t* scales,
                                                                          float* global, uint16_t* r_out) {
  __shared__ float s_ss[kMaxNormQThreads / 32];
  __shared__ float s_mx[kMaxNormQThreads / 32];
  __shared__ float s_peer[kMaxNormQRows];
  const uint32_t row = cluster_ctarank();
  const uint32_t csize = gridDim.x;          // the whole grid is one cluster
  if (csize > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  griddep_launch_dependents();
  const int nbr = K / 16;
  const int t = threadIdx.x, lane = t & 31, nw = blockDim.x >> 5;
  const bool live = t < nbr;
  const float* xb = x + (long)row * ld + (long)t * 16;
  if (live) prefetch_l2(xb);
  griddep_wait();                            // the input comes from the preceding kernel

  float v[16];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = 0.0f;
  if (live) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = __ldcg(reinterpret_cast<const float4*>(xb) + i);
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = __fmaf_rn(v[i], v[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) s_ss[t >> 5] = ss;
  __syncthreads();
  float tot = lane < nw ? s_ss[lane] : 0.0f;   // every warp reduces the same values the same way
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv = __fdiv_rn(1.0f, sqrtf(__fadd_rn(__fdiv_rn(tot, (float)K), eps)));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = round_bf16(__fmul_rn(v[i], inv));
  if (live && r_out) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = (__float_as_uint(v[2 * i]) >> 16) | (__float_as_uint(v[2 * i + 1]) & 0xFFFF0000u);
    uint4* dst = reinterpret_cast<uint4*>(r_out + (long)row * K + (long)t * 16);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  const float bm = block_absmax(v);          // 0 for the padding threads
  float amax = bm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_mx[t >> 5] = amax;
  __syncthreads();
  amax = lane < nw ? s_mx[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (csize > 1) {                           // as in quant_cluster_kernel
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (t < (int)csize) st_dsmem_f32(dsmem_addr(&s_peer[row], t), amax);
    cluster_sync();
    amax = lane < (int)csize ? s_peer[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  const float g = __fdiv_rn(amax, kGlobalDivisor);
  if (row == 0 && t == 0) *global = g;
  if (live) {
    uint2 c;
    const uint32_t sc = quant_block(v, bm, g, c);
    const long b = (long)row * nbr + t;
    reinterpret_cast<uint2*>(codes)[b] = c;
    scales[b] = static_cast<uint8_t>(sc);
  }
}

// ---- multi-launch path for large tensors -----------------------------------
template <class Src>
__global__ void __launch_bounds__(kThreads) amax_kernel(Src src, long nblocks, unsigned int* amax_bits) {
  __shared__ float s_warp[kThreads / 32];
  float local = 0.0f;
  for (long b = (long)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += (long)gridDim.x * kThreads) {
    float v[16];
    src.load(b, v);
    local = fmaxf(local, block_absmax(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local = fmaxf(local, __shfl_xor_sync(0xffffffffu, local, o));
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = local;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.0f;
    for (int w = 0; w < kThreads / 32; ++w) m = fmaxf(m, s_warp[w]);
    atomicMax(amax_bits, __float_as_uint(m));     // m >= 0: uint order == float order
  }
}

template <class Src>
__global__ void __launch_bounds__(kThreads) quant_grid_kernel(Src src, long nblocks, const float* amax,
                                                              uint8_t* codes, uint8_t* scales) {
  const float g = __fdiv_rn(*amax, kGlobalDivisor);
  for (long b = (long)blockIdx.x * kThreads + threadIdx.x; b < nblocks; b += (long)gridDim.x * kThreads) {
    float v[16];
    src.load(b, v);
    uint2 c;
    const uint32_t s = quant_block(v, block_absmax(v), g, c);
    reinterpret_cast<uint2*>(codes)[b] = c;
    scales[b] = static_cast<uint8_t>(s);
  }
}

__global__ void finalize_global_kernel(float* global) {
  *global = __fdiv_rn(*global, kGlobalDivisor);
}

__global__ void zero_global_kernel(float* global) { *global = 0.0f; }

// Largest cluster of quant_cluster_kernel<Src, NB> the current device can
// run (8, the portable size, or up to 16 with the non-portable opt-in, which
// this sets on the device).  Cached per device.
template <class Src, int NB>
int max_cluster() {
  static PerDeviceInt cap_cache;
  cudaError_t err = cudaSuccess;
  const int cap = cap_cache.get([](int, cudaError_t*) -> int {
    auto kern = quant_cluster_kernel<Src, NB>;
    int cap = 8;                                  // portable size, always available
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kMaxCluster);
      cfg.blockDim = dim3(kCThreads);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kMaxCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxPotentialClusterSize(&n, kern, &cfg) == cudaSuccess && n > cap) cap = n;
      if (cap > kMaxCluster) cap = kMaxCluster;
    }
    cudaGetLastError();
    return cap;
  }, &err);
  return cap > 0 ? cap : 8;
}

template <class Src, int NB>
cudaError_t launch_cluster(const Src& src, long nblocks, int csize, uint8_t* codes, uint8_t* scales,
                           float* global, cudaStream_t stream) {
  // Clusters above 8 CTAs need the non-portable opt-in, which max_cluster
  // sets on each device before it reports a cap above 8.
  if (csize > 8 && max_cluster<Src, NB>() < csize) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kCThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static const int trigger_late = [] {   // tuning knob: when the dependent GEMV may start launching
    const char* v = getenv("NVFP4_QUANT_TRIGGER");
    return (v && v[0] == 'l') ? 1 : 0;
  }();
  return cudaLaunchKernelEx(&cfg, quant_cluster_kernel<Src, NB>, src, nblocks, codes, scales, global, trigger_late);
}

template <class Src>
cudaError_t quantize_dispatch(const Src& src, long nblocks, uint8_t* codes, uint8_t* scales, float* global,
                              cudaStream_t stream) {
  if (nblocks == 0) {
    zero_global_kernel<<<1, 1, 0, stream>>>(global);
    return cudaGetLastError();
  }
  // One cluster: CTAs of kCThreads threads, each thread holding NB blocks in
  // registers; one block per thread while the device's cluster limit allows
  // (the work after the amax is a chain of IEEE divisions per block).
  const int cap = max_cluster<Src, 8>();
  if (nblocks <= (long)cap * kCThreads * 8) {
    long csize = (nblocks + kCThreads - 1) / kCThreads;
    if (csize < 1) csize = 1;
    if (csize > cap) csize = cap;
    const long T = csize * kCThreads;
    const long nb = (nblocks + T - 1) / T;
    if (nb <= 1) return launch_cluster<Src, 1>(src, nblocks, (int)csize, codes, scales, global, stream);
    if (nb <= 2) return launch_cluster<Src, 2>(src, nblocks, (int)csize, codes, scales, global, stream);
    if (nb <= 4) return launch_cluster<Src, 4>(src, nblocks, (int)csize, codes, scales, global, stream);
    return launch_cluster<Src, 8>(src, nblocks, (int)csize, codes, scales, global, stream);
  }
  int dev = 0, num_sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (num_sms <= 0) num_sms = 152;
  long grid = (nblocks + kThreads - 1) / kThreads;
  if (grid > (long)num_sms * 8) grid = (long)num_sms * 8;
  cudaError_t e = cudaMemsetAsync(global, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  amax_kernel<Src><<<(unsigned)grid, kThreads, 0, stream>>>(src, nblocks, reinterpret_cast<unsigned int*>(global));
  quant_grid_kernel<Src><<<(unsigned)grid, kThreads, 0, stream>>>(src, nblocks, global, codes, scales);
  finalize_global_kernel<<<1, 1, 0, stream>>>(global);
  return cudaGetLastError();
}

}  // namespace

// Defined in abi.cu.
nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);

extern "C" nvfp4_status nvfp4_quantize_act(const uint16_t* x_bf16, int rows, int K, uint8_t* codes,
                                           uint8_t* scales, float* global_scale, cudaStream_t stream) {
  if (rows < 0 || K < 0 || (K % 16) != 0) return NVFP4_ERR_SHAPE;
  if (!global_scale) return NVFP4_ERR_NULL;
  const long nblocks = (long)rows * (K / 16);
  if (nblocks > 0 && (!x_bf16 || !codes || !scales)) return NVFP4_ERR_NULL;
  if (!nvfp4_internal_aligned(x_bf16, 16) || !nvfp4_internal_aligned(codes, 16) ||
      !nvfp4_internal_aligned(scales, 4) || !nvfp4_internal_aligned(global_scale, 4))
    return NVFP4_ERR_ALIGN;
  SrcBF16 src{x_bf16, K / 16, K};
  return nvfp4_internal_cuda_status(quantize_dispatch(src, nblocks, codes, scales, global_scale, stream));
}

extern "C" nvfp4_status nvfp4_quantize_f32(const float* x, int rows, int K, int ld, uint8_t* codes,
                                           uint8_t* scales, float* global_scale, cudaStream_t stream) {
  if (rows < 0 || K < 0 || (K % 16) != 0 || ld < K || (ld % 4) != 0) return NVFP4_ERR_SHAPE;
  if (!global_scale) return NVFP4_ERR_NULL;
  const long nblocks = (long)rows * (K / 16);
  if (nblocks > 0 && (!x || !codes || !scales)) return NVFP4_ERR_NULL;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(codes, 16) ||
      !nvfp4_internal_aligned(scales, 4) || !nvfp4_internal_aligned(global_scale, 4))
    return NVFP4_ERR_ALIGN;
  SrcF32 src{x, K / 16, (long)ld};
  return nvfp4_internal_cuda_status(quantize_dispatch(src, nblocks, codes, scales, global_scale, stream));
}

extern "C" nvfp4_status nvfp4_silu_mul_quantize(const float* gate_up, int rows, int I, uint8_t* codes,
                                                uint8_t* scales, float* global_scale, cudaStream_t stream) {
  if (rows < 0 || I < 0 || (I % 16) != 0) return NVFP4_ERR_SHAPE;
  if (!global_scale) return NVFP4_ERR_NULL;
  const long nblocks = (long)rows * (I / 16);
  if (nblocks > 0 && (!gate_up || !codes || !scales)) return NVFP4_ERR_NULL;
  if (!nvfp4_internal_aligned(gate_up, 16) || !nvfp4_internal_aligned(codes, 16) ||
      !nvfp4_internal_aligned(scales, 4) || !nvfp4_internal_aligned(global_scale, 4))
    return NVFP4_ERR_ALIGN;
  SrcSiluMul src{gate_up, I / 16, I};
  return nvfp4_internal_cuda_status(quantize_dispatch(src, nblocks, codes, scales, global_scale, stream));
}

extern "C" nvfp4_status nvfp4_rms_norm_quantize(const float* x, int rows, int K, int ld, float eps, uint8_t* codes,
                                                uint8_t* scales, float* global_scale, uint16_t* r_out,
                                                cudaStream_t stream) {
  if (rows < 0 || K < 16 || (K % 16) != 0 || K / 16 > kMaxNormQThreads || ld < K || (ld % 4) != 0)
    return NVFP4_ERR_SHAPE;
  if (rows > kMaxNormQRows || !(eps >= 0.0f)) return NVFP4_ERR_RANGE;
  if (!global_scale) return NVFP4_ERR_NULL;
  if (rows > 0 && (!x || !codes || !scales)) return NVFP4_ERR_NULL;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(codes, 16) || !nvfp4_internal_aligned(scales, 4) ||
      !nvfp4_internal_aligned(global_scale, 4) || !nvfp4_internal_aligned(r_out, 16))
    return NVFP4_ERR_ALIGN;
  if (rows == 0) {
    zero_global_kernel<<<1, 1, 0, stream>>>(global_scale);
    return nvfp4_internal_cuda_status(cudaGetLastError());
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3((unsigned)(((K / 16) + 31) / 32 * 32));
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)rows;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return nvfp4_internal_cuda_status(cudaLaunchKernelEx(&cfg, rms_norm_quant_kernel, x, K, (long)ld, eps, codes, scales,
                                                       global_scale, r_out));
}
