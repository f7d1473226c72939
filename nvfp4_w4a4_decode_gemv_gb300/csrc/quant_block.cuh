// One 16-element block of the NVFP4 activation recipe (E4M3 block scale,
// E2M1 element codes), shared by the quantizer kernels and the GEMV that
// quantizes its activation in shared memory.  Format: ReSET reading note §2.1
// and §6.1 (E2M1 elements, E4M3 scale per 16-element block, FP32 global
// scale); every operation rounds once (IEEE), so the codes and the scale are
// those of a plain FP32 evaluation of
//   s = E4M3(bm / (6 g));  code = E2M1(x / (dec(s) g)).
#pragma once

#include "common.cuh"

namespace {

NVFP4_DEVINL float block_absmax(const float v[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// Quantize one block given the global scale g.  Returns the scale byte and
// writes the 8 code bytes.
NVFP4_DEVINL uint32_t quant_block(const float v[16], float bm, float g, uint2& codes) {
  const float d = __fmul_rn(6.0f, g);
  const float t = (d > 0.0f) ? __fdiv_rn(bm, d) : 0.0f;
  const uint32_t s = f32x2_to_e4m3x2(0.0f, t) & 0xFFu;
  const float S = __fmul_rn(e4m3_to_f32(s), g);
  // The code of v = x / S (IEEE quotient) is that of p = x * r with r = 1/S
  // (IEEE reciprocal) unless an E2M1 decision point (0.25, 0.75, ..., 5) lies
  // within the few ulps that separate p from v: |p - v| < 1.5 * 2^-23 |v|.  So
  // when the codes of p (1 - 2^-20) and p (1 + 2^-20) agree, every value in
  // between -- v among them -- has that code; otherwise divide.  All eight
  // pairs take the multiply path first, without branches, so that they
  // overlap; the divisions run only for the pairs (if any) left undecided.
  const float r = __frcp_rn(S);                 // +inf when S == 0 (codes are then sign-only)
  const bool fast = S > 0.0f && r < 1.0e38f;
  constexpr float kLo = 1.0f - 0x1.0p-20f, kHi = 1.0f + 0x1.0p-20f;
  uint32_t q[8];
  uint32_t undecided = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float pl = __fmul_rn(v[2 * i], r), ph = __fmul_rn(v[2 * i + 1], r);
    const uint32_t qa = f32x2_to_e2m1x2(__fmul_rn(ph, kLo), __fmul_rn(pl, kLo));
    const uint32_t qb = f32x2_to_e2m1x2(__fmul_rn(ph, kHi), __fmul_rn(pl, kHi));
    q[i] = qa;
    undecided |= (qa != qb ? 1u : 0u) << i;
  }
  if (!fast) undecided = (S > 0.0f) ? 0xFFu : 0u;
  if (undecided) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((undecided >> i) & 1u) q[i] = f32x2_to_e2m1x2(__fdiv_rn(v[2 * i + 1], S), __fdiv_rn(v[2 * i], S));
  }
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sgn = ((__float_as_uint(v[2 * i]) >> 31) << 3) | ((__float_as_uint(v[2 * i + 1]) >> 31) << 7);
    // magnitude from the conversion, sign from x; S == 0: the sign alone
    const uint32_t byte = (S > 0.0f) ? ((q[i] & 0x77u) | sgn) : sgn;
    packed[i >> 2] |= byte << (8 * (i & 3));
  }
  codes = make_uint2(packed[0], packed[1]);
  return s;
}

}  // namespace
