// Helpers for the kernels on the 5th-generation tensor cores (tcgen05, sm_103a):
// shared-memory matrix descriptors, MMA issue and commit, TMEM stores, and the
// Stream-K split shared by the GEMV and the prefill GEMM.
#pragma once

#include "common.cuh"

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
NVFP4_DEVINL uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

NVFP4_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
NVFP4_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (+)= A . B^T on 16-bit operands (kind::f16); acc = 0 overwrites D.
NVFP4_DEVINL void mma_f16(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(da), "l"(db), "r"(idesc), "r"(acc)
      : "memory");
}

// D (+)= (A x scales sfa) . (B x scales sfb)^T on E2M1 operands with one E4M3
// scale per 16 elements along K (kind::mxf4nvf4, scale_vec::4X).
NVFP4_DEVINL void mma_mxf4nvf4(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                               uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(da), "l"(db), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// One 32-bit column for the warp's 32 lanes.
NVFP4_DEVINL void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

NVFP4_DEVINL void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Bounded wait by a whole warp: lane 0 polls, the outcome is broadcast so that
// the warp stays converged (also when the wait gives up).
NVFP4_DEVINL bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Stream-K split: CTA q of G owns units [q U / G, (q+1) U / G).
NVFP4_DEVINL long long unit_start(long long q, long long U, long long G) { return (q * U) / G; }
NVFP4_DEVINL long long cta_of_unit(long long x, long long U, long long G) { return ((x + 1) * G - 1) / U; }
