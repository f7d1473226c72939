// Small-M NVFP4 W4A4 GEMV on CUDA cores (sm_103a):
//   y[m, n] = xg * wg * sum_k e2m1(x[m,k]) e4m3(sx[m,k/16]) e2m1(w[n,k]) e4m3(sw[n,k/16]),  M <= 8.
//
// The pages' design (ReSET project page, "Core contribution -- the nvfp4r
// CUDA-core kernel"; reading note §5.1-§5.2) streams each weight tile from
// HBM once and reuses it for every active token (C1), gives each thread
// several independent accumulator chains (C2) and dequantizes in registers
// with no shared-memory round trip of dequantized values and no CTA-wide
// synchronization in the K loop (C3).  This kernel keeps those three ideas and
// re-plans the rest for GB300:
//
//  * Weight tiles [128 rows x 256 K] (16 KB of codes + 2 KB of scales) are
//    moved HBM -> shared memory by TMA (cp.async.bulk.tensor, 128-byte
//    swizzle), issued by one producer warp into a ring of S stages guarded by
//    mbarriers (bounded waits).  Consumer warps read them with conflict-free
//    128-bit shared loads.  Only warp-level synchronization in the K loop.
//  * Each consumer lane owns R weight rows (C2) and all M tokens: R*M FP32
//    accumulators.  The activation operand of a 16-element block is a
//    warp-uniform 32-byte record (broadcast shared load) shared by the R rows.
//  * In-block products are exact integers: E2M1 values doubled are the
//    integers {0,1,2,3,4,6,8,12}; weights are mapped nibble -> (2v + 12) with
//    two byte-permute table lookups, activations to signed 2v, and __dp4a sums
//    four products per instruction.  The integer block sum lands in the
//    mantissa of 1.5 * 2^23 (exact for |sum| < 2^22), and one FMA removes that
//    offset while applying the activation block scale -- also exactly.  Across
//    blocks the sum is FP32: acc += (sx * D) * sw.
//  * Work is split Stream-K style: the [row tile x K chunk] units are cut into
//    equal contiguous ranges, one per CTA, so every SM streams the same number
//    of bytes whatever N and K are.  A row tile that two or more CTAs share is
//    finished by the last of them to arrive (an atomic counter per 32-row
//    sub-tile), which adds the partial sums in CTA order: deterministic, with
//    no spin-wait between CTAs.
//  * A small prep kernel turns the activation codes into the 32-byte records
//    (int8 values, bias-corrected dp4a seed, scale terms); it lets the GEMV
//    grid launch early (programmatic dependent launch), so the GEMV's first
//    weight TMAs overlap it.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

NVFP4_DEFINE_ERROR_READER(nvfp4_internal_read_error_gemv)

namespace {

constexpr int kChunk = 256;                 // K elements per stage
constexpr int kMaxM = 8;
constexpr int kRecBytes = 32;               // activation record per (token, 16-block)
constexpr int kRecsPerChunk = kChunk / 16;  // 16

// Weight nibble -> 12 + 2 * e2m1(code), split over two 8-entry tables for prmt.
// Positive codes index kPos*, negative codes (sign bit 3 flipped) index kNeg*.
constexpr uint32_t kPosLo = 0x0F0E0D0Cu, kPosHi = 0x18141210u;   // 12,13,14,15,16,18,20,24
constexpr uint32_t kNegLo = 0x090A0B0Cu, kNegHi = 0x00040608u;   // 12,11,10, 9, 8, 6, 4, 0

constexpr float kTwo58 = 288230376151711744.0f;          // 2^58
constexpr float kMagic = 12582912.0f;                    // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;

struct GemvArgs {
  const uint8_t* xrec;          // [C][M][16] records
  const float* xg;
  const float* wg;
  float* y;
  float* partials;              // [G][2][tile rows][M]
  unsigned int* counters;       // one per 32-row group of weight rows
  int M, N, K, C, RT;
  long long U;
};

NVFP4_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 8 weight nibbles (element i in bits 4i..4i+3) -> two words of biased bytes
// (element i in byte i of lo for i < 4, byte i - 4 of hi otherwise).
NVFP4_DEVINL void unpack_w8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t wx = w ^ 0x88888888u;
  lo = prmt(kPosLo, kPosHi, w) | prmt(kNegLo, kNegHi, wx);
  hi = prmt(kPosLo, kPosHi, w >> 16) | prmt(kNegLo, kNegHi, wx >> 16);
}


// ---- prep: activation codes -> records --------------------------------------
// Record of token m, block b: int8 x = 2*e2m1 (4 words, element i in byte i%4 of
// word i/4), dp4a seed c0 = 0x4B400000 - 12 * sum(x), sxs = e4m3(s) * 2^58,
// csx = -1.5*2^23 * sxs.  Stored at [(b / 16) * M + m][b % 16].
__global__ void __launch_bounds__(256) xrec_kernel(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs,
                                                   int M, int K, uint4* __restrict__ xrec) {
  griddep_launch_dependents();
  griddep_wait();               // the activation codes come from the preceding quantizer
  const int nb = K / 16;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M * nb) return;
  const int m = i / nb, b = i % nb;
  // L2-coherent loads: the codes come from the preceding kernel (see prefetch_l2).
  const uint2 cw = __ldcg(reinterpret_cast<const uint2*>(xq + (size_t)m * (K / 2)) + b);
  const uint32_t s = __ldcg(xs + (size_t)m * nb + b);
  uint32_t words[4] = {0u, 0u, 0u, 0u};
  int sum = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t c = ((e < 8 ? cw.x : cw.y) >> (4 * (e & 7))) & 15u;
    const int mag = (int)((0x0C08060403020100ull >> (8 * (c & 7u))) & 0xFFu);
    const int v = (c & 8u) ? -mag : mag;
    sum += v;
    words[e >> 2] |= ((uint32_t)v & 0xFFu) << (8 * (e & 3));
  }
  const float sxs = __fmul_rn(e4m3_to_f32(s), kTwo58);
  const float csx = __fmul_rn(-kMagic, sxs);
  uint4* dst = xrec + 2 * ((size_t)((b / kRecsPerChunk) * M + m) * kRecsPerChunk + (b % kRecsPerChunk));
  dst[0] = make_uint4(words[0], words[1], words[2], words[3]);
  dst[1] = make_uint4((uint32_t)(kMagicBits - 12 * sum), __float_as_uint(sxs), __float_as_uint(csx), 0u);
}

// ---- the GEMV kernel ----------------------------------------------------------
// Tile = TR weight rows x 256 K.  TR / (32 R) consumer warps, each lane owning R
// rows; one producer warp; S pipeline stages.
template <int M, int TR, int R>
struct Layout {
  static constexpr int kWC = TR / (32 * R);
  static_assert(kWC * 32 * R == TR && kWC >= 1, "tile rows must be a multiple of 32 R");
  static constexpr int kCodeBytes = TR * 128;          // one swizzled 128-byte row per weight row
  static constexpr int kScaleBytes = TR * 16;
  static constexpr int kXBytes = M * kRecsPerChunk * kRecBytes;
  static constexpr int kSlot = ((kCodeBytes + kScaleBytes + kXBytes + 1023) / 1024) * 1024;
};

template <int M, int TR, int R, int S>
constexpr size_t gemv_smem_bytes() {
  return (size_t)S * Layout<M, TR, R>::kSlot + 1024 /* alignment slack */ + 2 * S * sizeof(uint64_t);
}

NVFP4_DEVINL long long unit_start(long long q, long long U, long long G) { return (q * U) / G; }

// CTA whose unit range contains unit x: the largest q with unit_start(q) <= x.
NVFP4_DEVINL long long cta_of_unit(long long x, long long U, long long G) { return ((x + 1) * G - 1) / U; }

template <int R>
NVFP4_DEVINL float acc_get(const float2* a, int r) { return (r & 1) ? a[r / 2].y : a[r / 2].x; }

// One 256-K stage for this lane's R rows and all M tokens.  The block loop stays
// rolled (small code); the token and row loops are unrolled.
template <int M, int TR, int R>
NVFP4_DEVINL void compute_stage(const uint8_t* slot, int warp, int lane, float2 (&acc2)[M][(R + 1) / 2]) {
  using L = Layout<M, TR, R>;
  const uint8_t* codes = slot;
  const uint8_t* scl = slot + L::kCodeBytes;
  const uint4* xr = reinterpret_cast<const uint4*>(slot + L::kCodeBytes + L::kScaleBytes);
  int rr[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rr[r] = warp * 32 * R + r * 32 + lane;
#pragma unroll 1
  for (int j = 0; j < 8; ++j) {
    uint4 cw[R];
    uint32_t sb[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      cw[r] = *reinterpret_cast<const uint4*>(codes + rr[r] * 128 + ((j ^ (rr[r] & 7)) << 4));
      sb[r] = *reinterpret_cast<const unsigned short*>(scl + rr[r] * 16 + 2 * j);   // scales of blocks 2j, 2j+1
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int b = 2 * j + h;
      uint32_t wv[R][4];
      float swr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        unpack_w8(h ? cw[r].z : cw[r].x, wv[r][0], wv[r][1]);
        unpack_w8(h ? cw[r].w : cw[r].y, wv[r][2], wv[r][3]);
        swr[r] = __uint_as_float(((sb[r] >> (8 * h)) & 0xFFu) << 20);   // e4m3 * 2^-120
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint4 xa = xr[2 * (m * kRecsPerChunk + b)];
        const uint4 xb = xr[2 * (m * kRecsPerChunk + b) + 1];
        float t[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          int d = __dp4a((int)xa.x, (int)wv[r][0], (int)xb.x);
          d = __dp4a((int)xa.y, (int)wv[r][1], d);
          d = __dp4a((int)xa.z, (int)wv[r][2], d);
          d = __dp4a((int)xa.w, (int)wv[r][3], d);
          t[r] = fmaf(__int_as_float(d), __uint_as_float(xb.y), __uint_as_float(xb.z));   // exact: sx * D * 2^60
        }
#pragma unroll
        for (int r = 0; r + 1 < R; r += 2)
          acc2[m][r / 2] = __ffma2_rn(make_float2(t[r], t[r + 1]), make_float2(swr[r], swr[r + 1]), acc2[m][r / 2]);
        if (R & 1) acc2[m][R / 2].x = fmaf(t[R - 1], swr[R - 1], acc2[m][R / 2].x);
      }
    }
  }
}

template <int M, int TR, int R>
NVFP4_DEVINL void flush_tile(const GemvArgs& a, int tile, long long first_unit_of_cta, int warp, int lane,
                             const float2 (&acc2)[M][(R + 1) / 2]) {
  const long long G = gridDim.x;
  const long long C = a.C;
  const long long first = cta_of_unit((long long)tile * C, a.U, G);
  const long long last = cta_of_unit((long long)tile * C + C - 1, a.U, G);
  const float yscale = __fmul_rn(__fmul_rn(__ldcg(a.xg), __ldcg(a.wg)), 1152921504606846976.0f /* 2^60 */);
  const int row0 = tile * TR + warp * 32 * R;
  if (first == last) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int n = row0 + r * 32 + lane;
      if (n < a.N) {
#pragma unroll
        for (int m = 0; m < M; ++m) a.y[(size_t)m * a.N + n] = acc_get<R>(acc2[m], r) * yscale;
      }
    }
    return;
  }
  const int my_slot = (tile == (int)(first_unit_of_cta / C)) ? 0 : 1;
  float* part = a.partials + (((size_t)blockIdx.x * 2 + my_slot) * TR + warp * 32 * R) * M;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) __stcg(part + (size_t)(r * 32 + lane) * M + m, acc_get<R>(acc2[m], r));
  __syncwarp();                 // the warp's partial stores are ordered before lane 0's release
  unsigned int* cnt = a.counters + (size_t)(row0 / 32);
  int is_last = 0;
  if (lane == 0) {
    fence_acq_rel_gpu();        // release: this warp's partials before the count
    is_last = (atomicAdd(cnt, 1u) == (unsigned int)(last - first));
    if (is_last) fence_acq_rel_gpu();   // acquire: every contributor's partials
  }
  is_last = __shfl_sync(0xffffffffu, is_last, 0);
  if (!is_last) return;
  __syncwarp();                 // the lanes' partial loads are ordered after lane 0's acquire
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float sum[M];
#pragma unroll
    for (int m = 0; m < M; ++m) sum[m] = 0.0f;
    for (long long q = first; q <= last; ++q) {
      const int qslot = (tile == (int)(unit_start(q, a.U, G) / C)) ? 0 : 1;
      const float* pq = a.partials + (((size_t)q * 2 + qslot) * TR + warp * 32 * R + r * 32 + lane) * M;
#pragma unroll
      for (int m = 0; m < M; ++m) sum[m] += __ldcg(pq + m);
    }
    const int n = row0 + r * 32 + lane;
    if (n < a.N) {
#pragma unroll
      for (int m = 0; m < M; ++m) a.y[(size_t)m * a.N + n] = sum[m] * yscale;
    }
  }
  if (lane == 0) *cnt = 0u;
}

template <int M, int TR, int R, int S>
__global__ void __launch_bounds__(32 * (TR / (32 * R) + 1)) gemv_kernel(const __grid_constant__ CUtensorMap tm_codes,
                                                                        const __grid_constant__ CUtensorMap tm_scales,
                                                                        const GemvArgs a) {
  using L = Layout<M, TR, R>;
  constexpr int WC = L::kWC;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base for the 128-byte swizzle.  Offset arithmetic on the
  // shared array keeps every access in the shared state space.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * L::kSlot);
  uint64_t* empty = full + S;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const long long u0 = unit_start(blockIdx.x, a.U, G);
  const long long u1 = unit_start(blockIdx.x + 1, a.U, G);
  const int nunits = (int)(u1 - u0);
  constexpr uint32_t xbytes = (uint32_t)M * kRecsPerChunk * kRecBytes;
  constexpr uint32_t stage_tx = L::kCodeBytes + L::kScaleBytes + xbytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], WC);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) griddep_launch_dependents();   // the next kernel in the stream may start launching

  if (warp == WC) {
    // ---------------- producer warp ----------------
    if (lane == 0 && nunits > 0) {
      prefetch_tmap(&tm_codes);
      prefetch_tmap(&tm_scales);
      const int pre = nunits < S ? nunits : S;
      for (int k = 0; k < pre; ++k) {
        const long long u = u0 + k;
        const int tile = (int)(u / a.C), c = (int)(u % a.C);
        uint8_t* slot = smem + k * L::kSlot;
        mbar_arrive_expect_tx(&full[k], stage_tx);
        tma_load_2d(slot, &tm_codes, c * 128, tile * TR, &full[k]);
        tma_load_2d(slot + L::kCodeBytes, &tm_scales, c * 16, tile * TR, &full[k]);
      }
      griddep_wait();   // activation records are written by the prep kernel
      for (int k = 0; k < pre; ++k) {
        const int c = (int)((u0 + k) % a.C);
        bulk_g2s(smem + k * L::kSlot + L::kCodeBytes + L::kScaleBytes, a.xrec + (size_t)c * xbytes, xbytes, &full[k]);
      }
      int issued = pre;
      for (int k = pre; k < nunits; ++k) {
        const int s = k % S;
        if (!mbar_wait(&empty[s], ((k / S) - 1) & 1)) break;
        const long long u = u0 + k;
        const int tile = (int)(u / a.C), c = (int)(u % a.C);
        uint8_t* slot = smem + s * L::kSlot;
        mbar_arrive_expect_tx(&full[s], stage_tx);
        tma_load_2d(slot, &tm_codes, c * 128, tile * TR, &full[s]);
        tma_load_2d(slot + L::kCodeBytes, &tm_scales, c * 16, tile * TR, &full[s]);
        bulk_g2s(slot + L::kCodeBytes + L::kScaleBytes, a.xrec + (size_t)c * xbytes, xbytes, &full[s]);
        issued = k + 1;
      }
      // Do not leave the CTA with copies still in flight: wait (bounded) for the
      // last stages issued; on the normal path they have long completed.
      for (int k = (issued > S ? issued - S : 0); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    }
    return;
  }

  // ---------------- consumer warps ----------------
  griddep_wait();
  float2 acc2[M][(R + 1) / 2];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int r = 0; r < (R + 1) / 2; ++r) acc2[m][r] = make_float2(0.0f, 0.0f);
  int cur_tile = -1;
  for (int k = 0; k < nunits; ++k) {
    const int s = k % S;
    if (!mbar_wait(&full[s], (k / S) & 1)) return;    // error recorded; outputs incomplete
    const long long u = u0 + k;
    const int tile = (int)(u / a.C);
    if (tile != cur_tile) {
      if (cur_tile >= 0) flush_tile<M, TR, R>(a, cur_tile, u0, warp, lane, acc2);
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int r = 0; r < (R + 1) / 2; ++r) acc2[m][r] = make_float2(0.0f, 0.0f);
      cur_tile = tile;
    }
    compute_stage<M, TR, R>(smem + s * L::kSlot, warp, lane, acc2);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (cur_tile >= 0) flush_tile<M, TR, R>(a, cur_tile, u0, warp, lane, acc2);
}

// ---- host side ------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner_bytes, rows};
  const cuuint64_t strides[1] = {inner_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

constexpr int kMaxCtasPerSm = 8;
constexpr int kMaxTileRows = 128;

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t xrec, counters, tcrec, partials, total;
};

// Counters sit first, in a fixed-size region (one per 32-row group of weight
// rows), so that calls of any shape that share a workspace find them at the
// same place, and zero.
constexpr int kMaxN = 1 << 20;
constexpr size_t kCounterBytes = align256((size_t)(kMaxN / 32 + 64) * sizeof(unsigned int));

}  // namespace


// Defined in gemv_tc.cu.
size_t nvfp4_internal_tc_record_bytes();

namespace {

// [counters][records of the tensor-core path][activation records of the
// CUDA-core path][partial sums of the CUDA-core path].  The first two sit at
// fixed places (their size does not depend on the shape) because they must be
// zero at the start of every call, whatever the shape of the previous one.
WsLayout ws_layout(int M, int N, int K) {
  (void)N;
  WsLayout l;
  l.counters = 0;
  l.tcrec = kCounterBytes;
  l.xrec = l.tcrec + align256(nvfp4_internal_tc_record_bytes());
  l.partials = l.xrec + align256((size_t)M * (K / 16) * kRecBytes);
  const size_t gmax = (size_t)device_sms() * kMaxCtasPerSm;
  l.total = l.partials + align256(gmax * 2 * kMaxTileRows * (size_t)M * sizeof(float));
  return l;
}


template <int M, int TR, int R, int S>
cudaError_t launch_variant(const void* wq, const void* wsc, GemvArgs a, cudaStream_t stream, int grid_cap) {
  static PerDeviceInt occ_cache;
  constexpr int WC = TR / (32 * R);
  constexpr size_t smem = gemv_smem_bytes<M, TR, R, S>();
  auto kern = gemv_kernel<M, TR, R, S>;
  cudaError_t err = cudaSuccess;
  const int occ = occ_cache.get([](int, cudaError_t* e_out) -> int {
    auto k = gemv_kernel<M, TR, R, S>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int o = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k, 32 * (WC + 1), smem);
    if (e != cudaSuccess) {
      *e_out = e;
      return 0;
    }
    return o < 1 ? 1 : (o > kMaxCtasPerSm ? kMaxCtasPerSm : o);
  }, &err);
  if (occ == 0) return err;
  CUtensorMap tc, ts;
  if (!encode_2d(&tc, wq, (uint64_t)a.K / 2, (uint64_t)a.N, 128, TR, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&ts, wsc, (uint64_t)a.K / 16, (uint64_t)a.N, 16, TR, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  a.RT = (a.N + TR - 1) / TR;
  a.U = (long long)a.RT * a.C;
  long long G = (long long)occ * device_sms();
  if (grid_cap > 0 && G > grid_cap) G = grid_cap;
  if (G > a.U) G = a.U;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(32 * (WC + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tc, ts, a);
}

// Kernel variants: tile rows x rows per lane x pipeline stages.
template <int M>
cudaError_t launch_m(int variant, const void* wq, const void* wsc, const GemvArgs& a, cudaStream_t stream,
                     int grid_cap) {
  switch (variant) {
    case 1: return launch_variant<M, 128, 2, 3>(wq, wsc, a, stream, grid_cap);
    case 2: return launch_variant<M, 64, 1, 4>(wq, wsc, a, stream, grid_cap);
    case 3: return launch_variant<M, 64, 2, 4>(wq, wsc, a, stream, grid_cap);
    case 4: return launch_variant<M, 128, 1, 4>(wq, wsc, a, stream, grid_cap);
    case 5: return launch_variant<M, 64, 1, 6>(wq, wsc, a, stream, grid_cap);
    default: return launch_variant<M, 128, 1, 3>(wq, wsc, a, stream, grid_cap);
  }
}

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return v ? atoi(v) : dflt;
}

// Tuning knobs, read once per process: a grid cap for either GEMV kernel
// (NVFP4_GEMV_GRID, 0 = none) and the CUDA-core kernel's tile variant
// (NVFP4_GEMV_VARIANT).
int gemv_grid_cap() {
  static const int v = env_int("NVFP4_GEMV_GRID", 0);
  return v;
}
int gemv_variant() {
  static const int v = env_int("NVFP4_GEMV_VARIANT", 0);
  return v;
}

}  // namespace

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);
nvfp4_status nvfp4_internal_check_device();
cudaError_t nvfp4_internal_bf16_gemv_tc(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                                        unsigned int* records, cudaStream_t stream);
cudaError_t nvfp4_internal_gemv_tc(const uint8_t* xq, const uint8_t* xs, const float* xg, int M, const uint8_t* wq,
                                   const uint8_t* ws, const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                                   unsigned int* records, int grid_cap, int max_ctas_per_sm, cudaStream_t stream);
cudaError_t nvfp4_internal_quantize_gemv_tc(const uint16_t* x, int M, const uint8_t* wpacked, const float* wg, int N,
                                            int K, float* y, float* xg_out, unsigned int* records, int grid_cap,
                                            int max_ctas_per_sm, long long max_blocks, cudaStream_t stream,
                                            bool* launched);
cudaError_t nvfp4_internal_quantize_gemv_one_launch(int M, int N, int K, int grid_cap, int max_ctas_per_sm,
                                                    long long max_blocks, bool* one);
size_t nvfp4_internal_packed_bytes(int N, int K);
cudaError_t nvfp4_internal_pack_weights(const uint8_t* wq, const uint8_t* ws, int N, int K, uint8_t* packed,
                                        cudaStream_t stream);

bool nvfp4_internal_encode_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                              uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  return encode_2d(map, base, inner_bytes, rows, box_inner, box_rows,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

int nvfp4_internal_device_sms() { return device_sms(); }

void nvfp4_internal_test_gemv_fault(unsigned int flag_spin_limit, int drop_records);

extern "C" size_t nvfp4_gemv_workspace_bytes(int M, int N, int K) {
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return 0;
  return ws_layout(M, N, K).total;
}

namespace {
// Checks shared by the two row-major entry points.
nvfp4_status check_gemv_args(const uint8_t* xq, const uint8_t* xs, const float* xg, int M, const uint8_t* wq,
                             const uint8_t* ws, const float* wg, int N, int K, float* y, void* workspace,
                             size_t workspace_bytes) {
  if (!xq || !xs || !xg || !wq || !ws || !wg || !y || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxM) return NVFP4_ERR_RANGE;
  if (N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(xq, 16) || !nvfp4_internal_aligned(xs, 16) || !nvfp4_internal_aligned(wq, 16) ||
      !nvfp4_internal_aligned(ws, 16) || !nvfp4_internal_aligned(y, 16) || !nvfp4_internal_aligned(xg, 4) ||
      !nvfp4_internal_aligned(wg, 4) || !nvfp4_internal_aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  if (workspace_bytes < ws_layout(M, N, K).total) return NVFP4_ERR_SHAPE;
  return nvfp4_internal_check_device();
}
}  // namespace

extern "C" nvfp4_status nvfp4_gemv_smallm(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                          const uint8_t* wq, const uint8_t* ws, const float* wg, int N, int K,
                                          float* y, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const nvfp4_status st = check_gemv_args(xq, xs, xg, M, wq, ws, wg, N, K, y, workspace, workspace_bytes);
  if (st != NVFP4_OK) return st;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  return nvfp4_internal_cuda_status(nvfp4_internal_gemv_tc(
      xq, xs, xg, M, wq, ws, nullptr, wg, N, K, y,
      reinterpret_cast<unsigned int*>(wsb + ws_layout(M, N, K).tcrec), gemv_grid_cap(), kMaxCtasPerSm, stream));
}

// The CUDA-core kernel of this file: the pages' own design point, kept as an
// independent second implementation that the tests compare against.
extern "C" nvfp4_status nvfp4_gemv_smallm_cudacore(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                                   const uint8_t* wq, const uint8_t* ws, const float* wg, int N,
                                                   int K, float* y, void* workspace, size_t workspace_bytes,
                                                   cudaStream_t stream) {
  const nvfp4_status st = check_gemv_args(xq, xs, xg, M, wq, ws, wg, N, K, y, workspace, workspace_bytes);
  if (st != NVFP4_OK) return st;
  const WsLayout wl = ws_layout(M, N, K);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  GemvArgs a;
  a.xrec = wsb + wl.xrec;
  a.xg = xg;
  a.wg = wg;
  a.y = y;
  a.partials = reinterpret_cast<float*>(wsb + wl.partials);
  a.counters = reinterpret_cast<unsigned int*>(wsb + wl.counters);
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = K / kChunk;
  a.RT = 0;   // set by the variant (depends on its tile height)
  a.U = 0;

  const int nrec = M * (K / 16);
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3((nrec + 255) / 256);
  pcfg.blockDim = dim3(256);
  pcfg.stream = stream;
  cudaLaunchAttribute pattr[1];
  pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pattr[0].val.programmaticStreamSerializationAllowed = 1;
  pcfg.attrs = pattr;
  pcfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&pcfg, xrec_kernel, xq, xs, M, K, reinterpret_cast<uint4*>(wsb + wl.xrec));
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);

  const int variant = gemv_variant();
  const int grid_cap = gemv_grid_cap();
  switch (M) {
    case 1: e = launch_m<1>(variant, wq, ws, a, stream, grid_cap); break;
    case 2: e = launch_m<2>(variant, wq, ws, a, stream, grid_cap); break;
    case 3: e = launch_m<3>(variant, wq, ws, a, stream, grid_cap); break;
    case 4: e = launch_m<4>(variant, wq, ws, a, stream, grid_cap); break;
    case 5: e = launch_m<5>(variant, wq, ws, a, stream, grid_cap); break;
    case 6: e = launch_m<6>(variant, wq, ws, a, stream, grid_cap); break;
    case 7: e = launch_m<7>(variant, wq, ws, a, stream, grid_cap); break;
    default: e = launch_m<8>(variant, wq, ws, a, stream, grid_cap); break;
  }
  return nvfp4_internal_cuda_status(e);
}

extern "C" void nvfp4_test_gemv_fault(unsigned int flag_spin_limit, int drop_records) {
  nvfp4_internal_test_gemv_fault(flag_spin_limit, drop_records);
}

extern "C" size_t nvfp4_packed_weight_bytes(int N, int K) {
  if (N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return 0;
  return nvfp4_internal_packed_bytes(N, K);
}

extern "C" nvfp4_status nvfp4_pack_weights(const uint8_t* wq, const uint8_t* ws, int N, int K, uint8_t* packed,
                                           size_t packed_bytes, cudaStream_t stream) {
  if (!wq || !ws || !packed) return NVFP4_ERR_NULL;
  if (N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return NVFP4_ERR_SHAPE;
  if (packed_bytes < nvfp4_internal_packed_bytes(N, K)) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(wq, 16) || !nvfp4_internal_aligned(ws, 16) || !nvfp4_internal_aligned(packed, 16))
    return NVFP4_ERR_ALIGN;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  return nvfp4_internal_cuda_status(nvfp4_internal_pack_weights(wq, ws, N, K, packed, stream));
}

extern "C" nvfp4_status nvfp4_gemv_smallm_packed(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                                 const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!xq || !xs || !xg || !wpacked || !wg || !y || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxM) return NVFP4_ERR_RANGE;
  if (N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(xq, 16) || !nvfp4_internal_aligned(xs, 16) || !nvfp4_internal_aligned(wpacked, 16) ||
      !nvfp4_internal_aligned(y, 16) || !nvfp4_internal_aligned(xg, 4) || !nvfp4_internal_aligned(wg, 4) ||
      !nvfp4_internal_aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  const WsLayout wl = ws_layout(M, N, K);
  if (workspace_bytes < wl.total) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  return nvfp4_internal_cuda_status(nvfp4_internal_gemv_tc(
      xq, xs, xg, M, nullptr, nullptr, wpacked, wg, N, K, y, reinterpret_cast<unsigned int*>(wsb + wl.tcrec),
      gemv_grid_cap(), kMaxCtasPerSm, stream));
}

// The activation quantizer and the packed GEMV as one call.  One launch
// (the kernel quantizes the activation chunks each CTA needs, after reading
// the whole activation for its maximum) while M is at most the knob
// NVFP4_QGEMV_MAX_M, M * K at most NVFP4_QGEMV_MAX_MK, no CTA quantizes more
// than NVFP4_QGEMV_MAX_BLOCKS blocks and every CTA's chunks fit its shared
// memory; otherwise
// nvfp4_quantize_act into the workspace's tail, then the GEMV.
namespace {
int qgemv_max_mk() {
  static const int v = env_int("NVFP4_QGEMV_MAX_MK", 65536);
  return v;
}
// Blocks of 16 activation values one CTA may quantize (each CTA repeats the
// work for the chunks it uses, so past this the two launches are faster).
int qgemv_max_blocks() {
  static const int v = env_int("NVFP4_QGEMV_MAX_BLOCKS", 1024);
  return v;
}
// Tokens up to which the one-launch route is taken: every CTA reads the
// whole activation for its maximum, and past three tokens those reads cost
// more in a decode chain than the kernel boundary they remove.
int qgemv_max_m() {
  static const int v = env_int("NVFP4_QGEMV_MAX_M", 3);
  return v;
}
struct QgLayout {
  size_t codes, scales, global, total;
};
QgLayout qg_layout(int M, int N, int K) {
  QgLayout l;
  l.codes = ws_layout(M, N, K).total;
  l.scales = l.codes + align256((size_t)M * K / 2);
  l.global = l.scales + align256((size_t)M * K / 16);
  l.total = l.global + 256;
  return l;
}
}  // namespace

extern "C" size_t nvfp4_quantize_gemv_workspace_bytes(int M, int N, int K) {
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return 0;
  return qg_layout(M, N, K).total;
}

extern "C" int nvfp4_quantize_gemv_launches(int M, int N, int K) {
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return 0;
  if (!(M <= qgemv_max_m() && (long long)M * K <= (long long)qgemv_max_mk())) return 2;
  if (nvfp4_internal_check_device() != NVFP4_OK) return -1;
  bool one = false;
  if (nvfp4_internal_quantize_gemv_one_launch(M, N, K, gemv_grid_cap(), kMaxCtasPerSm, qgemv_max_blocks(), &one) !=
      cudaSuccess)
    return -1;
  return one ? 1 : 2;
}

extern "C" nvfp4_status nvfp4_quantize_gemv_packed(const uint16_t* x, int M, const uint8_t* wpacked, const float* wg,
                                                   int N, int K, float* y, float* xg_out, void* workspace,
                                                   size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !wpacked || !wg || !y || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxM) return NVFP4_ERR_RANGE;
  if (N < 1 || N > kMaxN || K < kChunk || (K % kChunk) != 0) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(wpacked, 16) || !nvfp4_internal_aligned(y, 16) ||
      !nvfp4_internal_aligned(wg, 4) || (xg_out && !nvfp4_internal_aligned(xg_out, 4)) ||
      !nvfp4_internal_aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  const QgLayout ql = qg_layout(M, N, K);
  if (workspace_bytes < ql.total) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  unsigned int* records = reinterpret_cast<unsigned int*>(wsb + ws_layout(M, N, K).tcrec);
  if (M <= qgemv_max_m() && (long long)M * K <= (long long)qgemv_max_mk()) {
    bool launched = false;
    const cudaError_t e = nvfp4_internal_quantize_gemv_tc(x, M, wpacked, wg, N, K, y, xg_out, records,
                                                          gemv_grid_cap(), kMaxCtasPerSm, qgemv_max_blocks(), stream,
                                                          &launched);
    if (e != cudaSuccess || launched) return nvfp4_internal_cuda_status(e);
  }
  uint8_t* xq = wsb + ql.codes;
  uint8_t* xs = wsb + ql.scales;
  float* xg = xg_out ? xg_out : reinterpret_cast<float*>(wsb + ql.global);
  const nvfp4_status qs = nvfp4_quantize_act(x, M, K, xq, xs, xg, stream);
  if (qs != NVFP4_OK) return qs;
  return nvfp4_internal_cuda_status(nvfp4_internal_gemv_tc(xq, xs, xg, M, nullptr, nullptr, wpacked, wg, N, K, y,
                                                           records, gemv_grid_cap(), kMaxCtasPerSm, stream));
}

// BF16 GEMV on the tensor-core kernel: it needs only the records region of a
// GEMV workspace (counters and records are at fixed places, so one workspace
// serves both kinds of call).
extern "C" size_t nvfp4_bf16_gemv_workspace_bytes(int M, int N, int K) {
  if (M < 1 || M > kMaxM || N < 1 || N > kMaxN || K < 64 || (K % 64) != 0) return 0;
  return ws_layout(M, N, kChunk).xrec;
}

extern "C" nvfp4_status nvfp4_bf16_gemv_tc(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !w || !y || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxM) return NVFP4_ERR_RANGE;
  if (N < 1 || N > kMaxN || K < 64 || (K % 64) != 0) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(x, 16) || !nvfp4_internal_aligned(w, 16) || !nvfp4_internal_aligned(y, 16) ||
      !nvfp4_internal_aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  const WsLayout wl = ws_layout(M, N, kChunk);
  if (workspace_bytes < wl.xrec) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  return nvfp4_internal_cuda_status(
      nvfp4_internal_bf16_gemv_tc(x, M, w, N, K, y, reinterpret_cast<unsigned int*>(wsb + wl.tcrec), stream));
}
