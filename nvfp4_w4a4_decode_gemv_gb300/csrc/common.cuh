// Device helpers shared by the sm_103a kernels of the NVFP4 decode library:
// status codes, bounded mbarrier waits, TMA bulk copies, cluster/DSMEM access.
//
// Every spin-wait here has an iteration limit.  A wait that runs out records
// an error code in the library's device status word and returns false; the
// caller then stops issuing work, waits (again bounded) for its own copies in
// flight and returns.  Nothing in this library traps or asserts on the device.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/nvfp4.h"

#define NVFP4_DEVINL __device__ __forceinline__

// Device-side error word, one per translation unit (internal linkage, so no
// relocatable device code is needed).  A bit set: kernels OR their error bits
// into it, so one error never erases another.  Every unit whose kernels set it
// defines a reader (NVFP4_DEFINE_ERROR_READER), and nvfp4_device_status()
// reads and clears them all.
static __device__ unsigned int g_nvfp4_device_error;

// Defines a host function that ORs this unit's error word into *out and
// clears it (synchronous copies).
#define NVFP4_DEFINE_ERROR_READER(fname)                                               \
  cudaError_t fname(unsigned int* out) {                                               \
    unsigned int v = 0, z = 0;                                                         \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_nvfp4_device_error, sizeof(v));         \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_nvfp4_device_error, &z, sizeof(z)); \
    *out |= v;                                                                         \
    return e;                                                                          \
  }

// Host: one positive int per device, computed by `compute(dev)` on the first
// call made with that device current.  Thread-safe: racing first calls compute
// the same value (and `compute` only sets attributes that are idempotent).
// A failed computation returns its error through *err and caches nothing.
struct PerDeviceInt {
  static constexpr int kMaxDevices = 64;
  std::atomic<int> v[kMaxDevices] = {};
  template <class F>
  int get(F compute, cudaError_t* err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    if (e != cudaSuccess) {
      *err = e;
      return 0;
    }
    int x = v[dev].load(std::memory_order_acquire);
    if (x > 0) return x;
    x = compute(dev, err);
    if (x > 0) v[dev].store(x, std::memory_order_release);
    return x;
  }
};

enum : unsigned int {
  NVFP4_DEVERR_NONE = 0,
  NVFP4_DEVERR_MBAR_TIMEOUT = 1,   // an mbarrier wait exceeded its iteration limit
  NVFP4_DEVERR_STATE_W = 2,        // reset_sample called with a window larger than the state's
  NVFP4_DEVERR_FLAG_TIMEOUT = 4,   // a wait for another CTA's partial sum exceeded its iteration limit
};

// Relaxed GPU-scope word store / load: single-copy atomic, no ordering.
NVFP4_DEVINL void st_relaxed_gpu(unsigned int* p, unsigned int v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
NVFP4_DEVINL unsigned int ld_relaxed_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ~ 2^26 polls of try_wait (each try_wait itself suspends for a while): seconds,
// far beyond any legitimate wait of these microsecond kernels.
constexpr uint32_t kMbarSpinLimit = 1u << 26;

NVFP4_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

NVFP4_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

NVFP4_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

NVFP4_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

NVFP4_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

NVFP4_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (and records the error) if the limit is reached.
NVFP4_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMbarSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_MBAR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
NVFP4_DEVINL void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled TMA load; coordinates in elements (x innermost).
NVFP4_DEVINL void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// GPU-scope acquire-release fence (cheaper than the sequentially consistent
// __threadfence).
NVFP4_DEVINL void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Programmatic dependent launch: wait for the preceding grid's completion and
// memory, and let the next grid start launching.
NVFP4_DEVINL void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
NVFP4_DEVINL void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Ask L2 for the line holding p.  A hint, but not an invisible one: when the
// line is rewritten afterwards (by a kernel still running while this one
// waits on it), a later non-coherent load (ld.global.nc) on this SM was
// measured to return the prefetched data.  Pair it with L2-coherent loads
// (ld.global.cg) only.
NVFP4_DEVINL void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

NVFP4_DEVINL void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---- clusters / distributed shared memory --------------------------------
NVFP4_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

NVFP4_DEVINL void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
NVFP4_DEVINL uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}

NVFP4_DEVINL void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---- number formats --------------------------------------------------------
// E4M3 byte (non-negative, finite) -> float, exactly: the 7 low bits placed at
// FP32 bits 26..20 give 2^-120 times the E4M3 value for normal and subnormal
// codes alike; the multiply by 2^120 is exact.
NVFP4_DEVINL float e4m3_to_f32(uint32_t s) {
  return __fmul_rn(__uint_as_float((s & 0x7Fu) << 20), __uint_as_float((127u + 120u) << 23) /* 2^120 */);
}

// RNE + saturating conversion of two non-negative floats to E4M3 bytes:
// returns (e4m3(hi) << 8) | e4m3(lo).
NVFP4_DEVINL uint32_t f32x2_to_e4m3x2(float hi, float lo) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// RNE + saturating conversion of two floats to E2M1: (e2m1(hi) << 4) | e2m1(lo).
NVFP4_DEVINL uint32_t f32x2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

NVFP4_DEVINL float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
NVFP4_DEVINL float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
