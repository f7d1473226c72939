// Small-M NVFP4 W4A4 GEMV on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same result as the CUDA-core kernel (gemv.cu):
//   y[m, n] = xg * wg * sum_k e2m1(x[m,k]) e4m3(sx[m,k/16]) e2m1(w[n,k]) e4m3(sw[n,k/16]).
//
// The pages reject tensor cores for decode because Blackwell's NVFP4 MMA tile
// is 128 rows along the token dimension, so at M <= 8 at most 8 of 128 rows do
// useful work (ReSET project page, "Why a CUDA-core NVFP4 kernel?"; reading
// note §5.1).  Swapping the operands removes that argument: the 128-row side
// of `tcgen05.mma ... kind::mxf4nvf4.block_scale.scale_vec::4X` takes 128
// WEIGHT rows, the tokens sit on the narrow N side (N = 16, M <= 8 used).  The
// tensor core then consumes the E2M1 codes and the E4M3 block scales as they
// are stored, so no CUDA-core instruction is spent per weight and the kernel
// is a pure HBM stream.  What the pages' design wanted -- every weight tile
// read from HBM once and used for every token (C1), no dequantized buffer (C3)
// -- holds here by construction.
//
// Per 256-K stage of a 128-row tile (one TMA ring slot):
//   producer warp   TMA: weight codes 128 x 128 B (128-byte swizzle), weight
//                   scales 128 x 16 B, token codes 16 x 128 B (swizzled; rows
//                   >= M arrive as zeros) and token scales 16 x 16 B.  The
//                   weight tiles of the first stages are issued before waiting
//                   on the preceding kernel (programmatic dependent launch), so
//                   they overlap the quantizer that produces the tokens.
//   4 scale warps   scale bytes -> TMEM with single-column stores.  An MMA
//                   whose weight-scale address is column A reads the 4 block
//                   scales of weight row r from lane r, column A + r/32 (one
//                   byte per 16-element block); with token-scale address B it
//                   reads token n's scales, for the accumulator rows of lane
//                   quadrant p, from lane 32p + n, column B.  So MMA q of a
//                   stage uses A = S0 + 4q, B = S1 + 4q; row r's word goes to
//                   column S0 + 4q + r/32, token n's word to lane 32p + n of
//                   column S1 + 4q in every quadrant p.
//   MMA thread      4 MMAs of K = 64 into a 128 x 16 FP32 TMEM accumulator;
//                   tcgen05.commit frees the slot
//   4 epilogue warps read the accumulator (double buffered) at tile ends and
//                   write y, or partial sums for the Stream-K fix-up
// Work split as in gemv.cu (Stream-K over [tile x 256-K] units); a split tile
// is finished by its first contributor (see the fix-up section below).
//
// The same kernel, instantiated with BF = true, is the BF16 GEMV of the
// lm_head (nvfp4_bf16_gemv_tc): `tcgen05.mma ... kind::f16` on BF16 operands,
// units of [128 rows x 64 K] (the same 128 bytes per row as an E2M1 unit, so
// the same swizzle, descriptor steps and ring), no scales and no output scale.
// Instantiated with QX = true it takes the BF16 activation and quantizes it
// itself (nvfp4_quantize_gemv_packed): the ring carries weights only, and the
// CTA's activation chunks stay in shared memory (qx_amax and qx_quant_chunk
// below).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "quant_block.cuh"
#include "tcgen05.cuh"

NVFP4_DEFINE_ERROR_READER(nvfp4_internal_read_error_gemv_tc)

namespace {

constexpr int kTR = 128;                    // weight rows per tile = MMA M
constexpr int kNT = 16;                     // MMA N: token rows (M <= 8 used, rest zero)
constexpr int kChunk = 256;                 // K per stage = 4 MMAs of K = 64
constexpr int kCodeBytes = kTR * 128;       // 16384
constexpr int kActCodeBytes = kNT * 128;    // 2048
constexpr int kActScaleBytes = kNT * 16;    // 256
constexpr int kScaleBytes = kTR * 16;       // 2048
constexpr int kActBytes = kActCodeBytes + kActScaleBytes;   // 2304: token codes + scales per stage
// slot: [A codes 16384][A scales 2048][B codes 2048][B scales 256], 1024-aligned slots.
// The first 18432 bytes are one block of the packed weight layout (see
// nvfp4_pack_weights), so a packed stage is one contiguous bulk copy.
constexpr int kOffSA = kCodeBytes;                          // 16384
constexpr int kOffB = kOffSA + kScaleBytes;                 // 18432 (1024-aligned: swizzled operand)
constexpr int kOffSB = kOffB + kActCodeBytes;               // 20480
constexpr int kSlot = ((kOffSB + kActScaleBytes + 1023) / 1024) * 1024;   // 21504
constexpr int kPackedBlock = kCodeBytes + kScaleBytes;      // 18432 bytes per [128-row tile x 256-K chunk]
constexpr uint32_t kStageTx = kCodeBytes + kScaleBytes + kActBytes;
constexpr int kWarps = 10;                  // 0 producer, 1 MMA, 2-5 scale writers, 6-9 epilogue
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kTmemCols = 256;         // D0 [0,16), D1 [16,32), D_last [32,48), 32 scale columns per stage (S <= 6)
constexpr uint32_t kColSF = 48;             // stage s: A scales at 48+32s+[0,16), B scales at 48+32s+16+[0,13)
// Instruction descriptor: E2M1 x E2M1 (format 1), UE4M3 scales, K-major A and B,
// N = 16 (bits 17-22: N >> 3), M = 128 (bits 24-28: M >> 4), dense.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kNT >> 3) << 17) | ((uint32_t)(kTR >> 4) << 24);
// BF16 operands (the lm_head variant, kind::f16): FP32 accumulator (bits 4-5 =
// 1), A and B both BF16 (bits 7-9 and 10-12 = 1), K-major, same N and M.
// A unit is [128 rows x 64 K] of BF16: 128 bytes per row, the same byte
// layout as an E2M1 unit, and the same 32-byte step per MMA (K = 16).
constexpr uint32_t kIdescBF16 =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kNT >> 3) << 17) | ((uint32_t)(kTR >> 4) << 24);
constexpr uint32_t kStageTxBF16 = kCodeBytes + kActCodeBytes;

// Activation quantized in the kernel (nvfp4_quantize_gemv_packed).  The ring
// slots carry weights only (one packed block); the CTA's activation chunks
// stay in shared memory for the whole call: chunk i's token codes are one
// 128-byte-swizzled atom of 8 rows at res + 1024 i (rows >= M zero), so the
// MMA's 16-row B operand reads rows 8-15 from the next atom -- accumulator
// columns 8-15, which nothing reads -- and an extra zero atom follows the
// last chunk; chunk i's token scales are 16 rows x 16 bytes at res_sc + 256 i.
constexpr int kSlotQX = kPackedBlock;       // 18432, 1024-aligned
constexpr int kMaxRes = 24;                 // activation chunks a CTA may hold
constexpr int kResCodeBytes = (kMaxRes + 1) * 1024;
constexpr int kResScaleBytes = kMaxRes * 256;
constexpr int kQThreads = 256;              // warps 2-9 quantize

struct TcArgs {
  const uint8_t* wpacked;        // packed weights, or null: weights through the two tensor maps
  const float* xg;
  const float* wg;
  float* y;
  unsigned int* records;         // [G][M][128] words: a CTA's partial sums of its first tile; zero between calls
  const uint16_t* x;             // QX: BF16 activation [M, K]
  float* xg_out;                 // QX: receives the activation's global scale (may be null)
  int M, N, K, C, RT;
  long long U;                   // units = RT * C, numbered tile-major
  uint32_t flag_spins;           // polls of a record before the wait gives up (kFlagSpinLimit)
  int drop_records;              // test hook: non-zero = publish no record (the first contributor's wait runs out)
};

// ---- Stream-K fix-up ---------------------------------------------------------------
// A tile that one CTA covers whole goes straight to y.  A split tile's
// contributors are the consecutive CTAs `first` .. `last`.  For every one but
// the first the tile is the first of its range: it writes its partial sums to
// its record and is done.  For the first the tile is the last of its range: it
// adds the others' records, in CTA order, to its own sums and writes y.
// A record word holds the bitwise complement of an FP32 partial sum; a finite
// value never encodes to zero, so a word is ready once it is non-zero and needs
// no flag, counter or fence, and the reader puts the zero back.  Records are
// therefore zero between calls, and the order of the additions is fixed by
// the split alone, so the result does not depend on timing.
constexpr uint32_t kFlagSpinLimit = 1u << 24;

struct Split {                  // a tile's contributors
  long long first, last;
  bool whole;
};

NVFP4_DEVINL Split split_of(const TcArgs& a, int tile, long long G) {
  Split sp;
  const long long C = a.C, t0 = (long long)tile * C;
  sp.first = cta_of_unit(t0, a.U, G);
  sp.last = cta_of_unit(t0 + C - 1, a.U, G);
  sp.whole = sp.first == sp.last;
  return sp;
}

// The output scale xg * wg (1 for BF16).  Read once per thread right after the
// dependency wait, off the critical path of the tile ends; L2-coherent loads,
// as xg comes from the preceding kernel (see prefetch_l2).
template <bool BF>
NVFP4_DEVINL float output_scale(const TcArgs& a) {
  return BF ? 1.0f : __fmul_rn(__ldcg(a.xg), __ldcg(a.wg));
}

template <int M>
NVFP4_DEVINL void store_y(const TcArgs& a, float yscale, int tile, int row, const float (&v)[kNT]) {
  const int n = tile * kTR + row;
  if (n < a.N) {
#pragma unroll
    for (int m = 0; m < M; ++m) a.y[(size_t)m * a.N + n] = v[m] * yscale;
  }
}

template <int M>
NVFP4_DEVINL unsigned int* record(const TcArgs& a, long long q, int row) {
  return a.records + (size_t)q * (size_t)(M * kTR) + row;
}

// A contributor other than the first: its partial sums, encoded.
template <int M>
NVFP4_DEVINL void publish_record(const TcArgs& a, int row, const float (&acc)[kNT]) {
  if (a.drop_records) return;
  unsigned int* rec = record<M>(a, blockIdx.x, row);
#pragma unroll
  for (int m = 0; m < M; ++m) st_relaxed_gpu(rec + m * kTR, ~__float_as_uint(acc[m]));
}

// The records of contributors q0 .. q0+3 (those <= last), once every word is
// written (bounded wait); every live word is then reset to zero.  A wait that
// gives up sets device error bit 2 and zeroes the words all the same, so a
// record published late is the only thing it can leave behind (the caller
// re-zeroes the workspace after that error).
template <int M>
NVFP4_DEVINL void take_records(const TcArgs& a, long long q0, long long last, int row, float (&v)[4][M]) {
  unsigned int w[4][M];
  // Every live word's load is issued before any is looked at (the loads are
  // ordered asm statements: a check between them would wait out each one's
  // L2 round trip in turn); only the words still zero are polled again.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool live = q0 + i <= last;
    const unsigned int* rec = record<M>(a, live ? q0 + i : q0, row);
#pragma unroll
    for (int m = 0; m < M; ++m) w[i][m] = live ? ld_relaxed_gpu(rec + m * kTR) : ~0u;
  }
  uint32_t spins = 0;
  for (;;) {
    bool ready = true;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < M; ++m) ready = ready && w[i][m] != 0u;
    if (ready) break;
    if (++spins >= a.flag_spins) {
      atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_FLAG_TIMEOUT);
      break;
    }
    __nanosleep(32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const unsigned int* rec = record<M>(a, q0 + i <= last ? q0 + i : q0, row);
#pragma unroll
      for (int m = 0; m < M; ++m)
        if (w[i][m] == 0u) w[i][m] = ld_relaxed_gpu(rec + m * kTR);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool live = q0 + i <= last;
    unsigned int* rec = record<M>(a, live ? q0 + i : q0, row);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      v[i][m] = __uint_as_float(~w[i][m]);
      if (live) st_relaxed_gpu(rec + m * kTR, 0u);
    }
  }
}

// Read a quadrant's 16 accumulator columns of buffer d, then release the buffer.
NVFP4_DEVINL void read_acc(uint32_t tmem, int quad, int d, uint64_t* acc_empty_d, float (&acc)[kNT]) {
  uint32_t r[kNT];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(d * kNT)));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && acc_empty_d) mbar_arrive(acc_empty_d);
#pragma unroll
  for (int i = 0; i < kNT; ++i) acc[i] = __uint_as_float(r[i]);
}

NVFP4_DEVINL void qx_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kQThreads) : "memory"); }

// The activation quantizer inside the GEMV (QX).
// * qx_amax (warps 2-9): every CTA reads the whole BF16 activation for the
//   tensor maximum -- so no CTA waits for another -- and forms the global
//   scale amax / 2688 as nvfp4_quantize_act does.
// * qx_quant_chunk (warps 6-9, the epilogue warps, idle until the first tile
//   ends): the nres chunks the CTA uses (chunk0, chunk0 + 1, ... mod C), warp
//   6 + q taking chunks q, q + 4, ..., each into its resident atom and scale
//   row with the recipe's roundings (quant_block), so the codes are the ones
//   nvfp4_quantize_act writes.  Chunk i's mbarrier completes when its codes
//   are in place; the scale writers wait for it before the chunk's first
//   unit, so only the first chunk sits on the path to the first MMA, and the
//   others are quantized while the weights stream.  (Chunk 0 shared by all
//   eight warps, one block a thread, measured slower: 0.538 against 0.529 ms
//   for the sweep's step.)
constexpr int kQF = 4;                       // blocks of one chunk a quantizing lane holds (M * 16 / 32)

// Chunk i's blocks of x: lane l holds blocks l, l + 32, ... of the chunk's
// M x 16 (block j of token m is number 16 m + j), two 16-byte pieces each.
template <int M>
NVFP4_DEVINL void qx_load_chunk(const TcArgs& a, int i, int chunk0, int lane, uint4 (&r)[kQF][2]) {
  int c = chunk0 + i;
  if (c >= a.C) c -= a.C;
#pragma unroll
  for (int u = 0; u < kQF; ++u) {
    const int b = lane + 32 * u;
    if (b < M * 16) {
      const uint4* p = reinterpret_cast<const uint4*>(a.x + (size_t)(b >> 4) * a.K + (size_t)c * kChunk +
                                                      (size_t)(b & 15) * 16);
      r[u][0] = __ldcg(p);
      r[u][1] = __ldcg(p + 1);
    }
  }
}

// Block j of token m of resident chunk i (16 BF16 values) into its atom and scale row.
NVFP4_DEVINL void qx_quant_block(uint8_t* res, uint8_t* res_sc, int i, int m, int j, const uint4 (&r)[2], float g) {
  const uint32_t w[8] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w};
  float v[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    v[2 * e] = bf16_lo(w[e]);
    v[2 * e + 1] = bf16_hi(w[e]);
  }
  uint2 codes;
  const uint32_t sc = quant_block(v, block_absmax(v), g, codes);
  // row m of the atom: 16-byte piece p at m*128 + ((p ^ m) * 16), as the TMA's
  // 128-byte swizzle places it; block j is the half (j & 1) of piece j/2.
  *reinterpret_cast<uint2*>(res + i * 1024 + m * 128 + ((((j >> 1) ^ m) & 7) << 4) + (j & 1) * 8) = codes;
  res_sc[i * 256 + m * 16 + j] = static_cast<uint8_t>(sc);
}

template <int M>
NVFP4_DEVINL void qx_quant_chunk(uint8_t* res, uint8_t* res_sc, int i, int lane, const uint4 (&r)[kQF][2],
                                 float g) {
#pragma unroll
  for (int u = 0; u < kQF; ++u) {
    const int b = lane + 32 * u;
    if (b < M * 16) qx_quant_block(res, res_sc, i, b >> 4, b & 15, r[u], g);
  }
}

// Warps 2-9.  Warps 6-9 also load the first chunk they quantize (into
// `first`) right after the dependency wait, with the maximum's loads.
template <int M>
NVFP4_DEVINL float qx_amax(const TcArgs& a, uint8_t* res, uint8_t* res_sc, uint32_t* s_wmax, int nres, int chunk0,
                           uint4 (&first)[kQF][2]) {
  const int qt = (int)threadIdx.x - 64;      // 0 .. 255
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int xbytes = M * a.K * 2;
  // While the preceding kernel may still run: zero the atoms (rows >= M and
  // the trailing atom stay zero) and the scale rows, and ask L2 for x.
  for (int o = qt * 16; o < (nres + 1) * 1024; o += kQThreads * 16)
    *reinterpret_cast<uint4*>(res + o) = make_uint4(0u, 0u, 0u, 0u);
  for (int o = qt * 16; o < nres * 256; o += kQThreads * 16)
    *reinterpret_cast<uint4*>(res_sc + o) = make_uint4(0u, 0u, 0u, 0u);
  for (int o = qt * 128; o < xbytes; o += kQThreads * 128) prefetch_l2(reinterpret_cast<const uint8_t*>(a.x) + o);
  griddep_wait();                            // x comes from the preceding kernel
  if (warp >= 6 && warp - 6 < nres) qx_load_chunk<M>(a, warp - 6, chunk0, lane, first);
  // max |x| over the tensor.  For BF16 magnitudes (sign cleared) the unsigned
  // order of the bit patterns is the order of the values, so the maximum is
  // taken on the bits, two halves at a time.
  const uint4* x4 = reinterpret_cast<const uint4*>(a.x);
  const int n4 = xbytes / 16;
  uint32_t mx = 0u;
  for (int b = qt; b < n4; b += kQThreads * 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = b + u * kQThreads;
      v[u] = i < n4 ? __ldcg(x4 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      mx = __vmaxu2(mx, v[u].x & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, v[u].y & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, v[u].z & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, v[u].w & 0x7FFF7FFFu);
    }
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) s_wmax[qt >> 5] = mx;
  qx_barrier();                              // also orders the zeroing before every code store
  uint32_t m8 = lane < kQThreads / 32 ? s_wmax[lane] : 0u;
  m8 = __reduce_max_sync(0xffffffffu, m8);
  const float g = __fdiv_rn(__uint_as_float(m8 << 16), 2688.0f);   // 448 * 6
  if (blockIdx.x == 0 && qt == 0 && a.xg_out) *a.xg_out = g;
  return g;
}

template <int M, int S, bool BF, bool QX = false>
__global__ void __launch_bounds__(kThreads, 2) gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_codes,
                                                              const __grid_constant__ CUtensorMap tm_scales,
                                                              const __grid_constant__ CUtensorMap tm_xcodes,
                                                              const __grid_constant__ CUtensorMap tm_xscales,
                                                              const TcArgs a) {
  static_assert(S >= 2 && kColSF + 32 * S <= kTmemCols, "scale columns must fit the TMEM allocation");
  static_assert(!(QX && BF), "the in-kernel quantizer produces NVFP4 operands");
  constexpr int kSl = QX ? kSlotQX : kSlot;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* res = smem + S * kSl;                        // QX: resident activation atoms
  uint8_t* res_sc = res + kResCodeBytes;                // QX: their token scale rows
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kSl + (QX ? kResCodeBytes + kResScaleBytes : 0));
  uint64_t* sf_ready = full + S;
  uint64_t* empty = sf_ready + S;
  uint64_t* acc_full = empty + S;           // [0], [1]: alternating tiles; [2]: the CTA's last tile
  uint64_t* acc_empty = acc_full + 3;
  uint64_t* chunk_ready = acc_empty + 2;                // QX: [kMaxRes] resident chunk i quantized
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(chunk_ready + (QX ? kMaxRes : 0));
  uint32_t* s_wmax = tmem_slot + 4;                     // QX: the quantizing warps' maxima

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const long long u0 = unit_start(blockIdx.x, a.U, G);
  const long long u1 = unit_start(blockIdx.x + 1, a.U, G);
  const int nunits = (int)(u1 - u0);
  const int nres = nunits < a.C ? nunits : a.C;         // QX: activation chunks this CTA uses (<= kMaxRes)

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sf_ready[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int d = 0; d < 3; ++d) mbar_init(&acc_full[d], 1);
    for (int d = 0; d < 2; ++d) mbar_init(&acc_empty[d], 4);
    if (QX)
      for (int i = 0; i < kMaxRes; ++i) mbar_init(&chunk_ready[i], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();   // the next kernel in the stream may start launching

  // Every role walks the CTA's units u0 .. u1-1 in order, keeping the unit's
  // (tile, chunk) and its ring slot and phase incrementally: no division in the loops.
  const int C = a.C;
  const int tile0 = (int)(u0 / C), chunk0 = (int)(u0 % C);

  // QX: warps 2-9 find the global scale; then warps 6-9 quantize the chunks,
  // each signalling its chunk's mbarrier, and go on to the epilogue.  The
  // scale writers wait for a chunk before its first unit, so their arrival on
  // sf_ready (which the MMA waits for) follows the chunk's codes.
  float qg = 0.0f;
  if (QX && warp >= 2 && nunits > 0) {
    uint4 first[kQF][2];
    qg = qx_amax<M>(a, res, res_sc, s_wmax, nres, chunk0, first);
    if (warp >= 6) {
      for (int i = warp - 6; i < nres; i += 4) {
        if (i != warp - 6) qx_load_chunk<M>(a, i, chunk0, lane, first);
        qx_quant_chunk<M>(res, res_sc, i, lane, first, qg);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the MMA reads the atom via the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&chunk_ready[i]);
      }
    }
  }

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0 && nunits > 0) {
      constexpr uint32_t tx = QX ? (uint32_t)kPackedBlock : BF ? kStageTxBF16 : kStageTx;
      if (!a.wpacked) {
        prefetch_tmap(&tm_codes);
        if (!BF) prefetch_tmap(&tm_scales);
      }
      if (!QX) {
        prefetch_tmap(&tm_xcodes);
        if (!BF) prefetch_tmap(&tm_xscales);
      }
      const int pre = nunits < S ? nunits : S;
      const uint8_t* wp = a.wpacked ? a.wpacked + (size_t)u0 * kPackedBlock : nullptr;
      // Weight tiles do not depend on the preceding kernel: issue the first
      // stages before waiting on it.
      {
        int tile = tile0, c = chunk0;
        for (int k = 0; k < pre; ++k) {
          uint8_t* slot = smem + k * kSl;
          mbar_arrive_expect_tx(&full[k], tx);
          if (wp) {
            bulk_g2s(slot, wp + (size_t)k * kPackedBlock, kPackedBlock, &full[k]);
          } else {
            tma_load_2d(slot, &tm_codes, c * 128, tile * kTR, &full[k]);
            if (!BF) tma_load_2d(slot + kOffSA, &tm_scales, c * 16, tile * kTR, &full[k]);
          }
          if (++c == C) { c = 0; ++tile; }
        }
      }
      int tile = tile0, c = chunk0;
      if (!QX) {               // (QX: the activation is quantized in this CTA; weights only here)
        griddep_wait();        // the token codes and scales come from the preceding kernel
        for (int k = 0; k < pre; ++k) {
          uint8_t* slot = smem + k * kSlot;
          tma_load_2d(slot + kOffB, &tm_xcodes, c * 128, 0, &full[k]);      // rows >= M arrive as zeros
          if (!BF) tma_load_2d(slot + kOffSB, &tm_xscales, c * 16, 0, &full[k]);
          if (++c == C) { c = 0; ++tile; }
        }
      } else {
        for (int k = 0; k < pre; ++k)
          if (++c == C) { c = 0; ++tile; }
      }
      int issued = pre;
      int s = pre % S;
      uint32_t phase = (pre / S) & 1;                    // phase of the slot's next fill
      for (int k = pre; k < nunits; ++k) {
        if (!mbar_wait(&empty[s], phase ^ 1u)) break;   // the slot's previous use has been consumed
        uint8_t* slot = smem + s * kSl;
        mbar_arrive_expect_tx(&full[s], tx);
        if (wp) {
          bulk_g2s(slot, wp + (size_t)k * kPackedBlock, kPackedBlock, &full[s]);
        } else {
          tma_load_2d(slot, &tm_codes, c * 128, tile * kTR, &full[s]);
          if (!BF) tma_load_2d(slot + kOffSA, &tm_scales, c * 16, tile * kTR, &full[s]);
        }
        if (!QX) {
          tma_load_2d(slot + kOffB, &tm_xcodes, c * 128, 0, &full[s]);
          if (!BF) tma_load_2d(slot + kOffSB, &tm_xscales, c * 16, 0, &full[s]);
        }
        issued = k + 1;
        if (++c == C) { c = 0; ++tile; }
        if (++s == S) { s = 0; phase ^= 1u; }
      }
      // Do not leave the CTA with copies still in flight: wait (bounded) for the
      // last stages issued; on the normal path they have long completed.
      for (int k = (issued > S ? issued - S : 0); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0 && nunits > 0) {
      // Descriptors of slot 0; the start-address field (bits 0-13, address / 16)
      // moves by (slot offset + 32 q) / 16 within the 14-bit field.
      const uint64_t da0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t db0 = smem_desc_sw128(smem_u32(QX ? res : smem + kOffB));
      // The CTA's last tile accumulates in its own buffer (D_last), flushed by
      // the scale writers; the others alternate between D0 and D1.
      const int last_idx = (int)((u1 - 1) / C) - tile0;
      int tile_idx = -1;
      int c = chunk0;
      int s = 0;
      uint32_t phase = 0;
      int issued = 0;
      int ri = 0;                                        // QX: resident chunk of the unit
      uint32_t d_tmem = tmem;
      for (int k = 0; k < nunits; ++k) {
        const bool first_of_tile = (k == 0) || (c == 0);
        if (first_of_tile) {
          ++tile_idx;
          if (tile_idx == last_idx) {
            d_tmem = tmem + (uint32_t)(2 * kNT);
          } else {
            if (tile_idx >= 2 && !mbar_wait(&acc_empty[tile_idx & 1], ((tile_idx >> 1) - 1) & 1)) break;
            d_tmem = tmem + (uint32_t)((tile_idx & 1) * kNT);
          }
        }
        // The scale writers arrive on sf_ready only after they have seen the
        // slot full, so sf_ready also orders the slot's data before the MMAs.
        // BF16 has no scales: the MMA waits for the slot itself.
        if (!mbar_wait(BF ? &full[s] : &sf_ready[s], phase)) break;
        tc_fence_after();
        const uint64_t doff = (uint64_t)((s * kSl) >> 4);
        const uint64_t dboff = QX ? (uint64_t)(ri * (1024 >> 4)) : doff;
        const uint32_t sfa = tmem + kColSF + 32u * s;
        const uint32_t sfb = sfa + 16u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (BF)
            mma_f16(d_tmem, da0 + doff + 2 * q, db0 + doff + 2 * q, kIdescBF16, (first_of_tile && q == 0) ? 0u : 1u);
          else
            mma_mxf4nvf4(d_tmem, da0 + doff + 2 * q, db0 + dboff + 2 * q, kIdesc, sfa + 4u * q, sfb + 4u * q,
                         (first_of_tile && q == 0) ? 0u : 1u);
        }
        mma_commit(&empty[s]);
        issued = k + 1;
        if (QX && ++ri == C) ri = 0;
        if (++c == C) c = 0;
        if (k + 1 == nunits || c == 0)                                          // last unit of this tile
          mma_commit(&acc_full[tile_idx == last_idx ? 2 : (tile_idx & 1)]);
        if (++s == S) { s = 0; phase ^= 1u; }
      }
      // Do not leave with MMAs in flight: wait (bounded) for the last commit.
      if (issued > 0) mbar_wait(&empty[(issued - 1) % S], ((issued - 1) / S) & 1);
    }
  } else if (warp < 6) {
    // ---------------- scale writers: rows 32*quad .. 32*quad + 31 ----------------
    // Their first slot holds token scales of the preceding kernel anyway, so
    // waiting on that kernel here costs nothing, and the output scale's load
    // overlaps the whole stream.
    griddep_wait();
    const float yscale = QX ? __fmul_rn(qg, __ldcg(a.wg)) : output_scale<BF>(a);
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t ta0 = tmem + ((uint32_t)(quad * 32) << 16) + kColSF + (uint32_t)quad;
    const uint32_t tb0 = tmem + ((uint32_t)(quad * 32) << 16) + kColSF + 16u;
    int s = 0;
    uint32_t phase = 0;
    int ri = 0;                                        // QX: resident chunk of the unit
    for (int k = 0; k < (BF ? 0 : nunits); ++k) {     // BF16 has no scales to place
      if (!mbar_wait_warp(&full[s], phase)) break;
      if (QX && k < nres && !mbar_wait_warp(&chunk_ready[ri], 0)) break;   // the unit's chunk, on its first use
      const uint8_t* slot = smem + s * kSl;
      const uint4 sa = *reinterpret_cast<const uint4*>(slot + kOffSA + row * 16);
      const uint32_t ta = ta0 + 32u * s;
      tmem_st1(ta, sa.x);
      tmem_st1(ta + 4u, sa.y);
      tmem_st1(ta + 8u, sa.z);
      tmem_st1(ta + 12u, sa.w);
      // Token scales: the MMA reads token n's scales for accumulator rows of
      // quadrant p from lane 32p + n, so every quadrant holds a copy.
      uint4 sb = make_uint4(0u, 0u, 0u, 0u);
      if (lane < kNT) sb = *reinterpret_cast<const uint4*>(QX ? res_sc + ri * 256 + lane * 16 : slot + kOffSB + lane * 16);
      if (QX && ++ri == C) ri = 0;
      const uint32_t tb = tb0 + 32u * s;
      tmem_st1(tb, sb.x);
      tmem_st1(tb + 4u, sb.y);
      tmem_st1(tb + 8u, sb.z);
      tmem_st1(tb + 12u, sb.w);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_ready[s]);
      if (++s == S) { s = 0; phase ^= 1u; }
    }
    // The CTA's last tile is flushed here, by warps that are idle once the
    // scales are written, so it does not wait behind the earlier tiles' flushes.
    if (nunits > 0) {
      const int tile_last = (int)((u1 - 1) / C);
      const int row = quad * 32 + lane;
      const Split sp = split_of(a, tile_last, G);
      const bool fin = !sp.whole && sp.first == (long long)blockIdx.x;   // this CTA finishes the tile
      float pre[4][M];
      if (fin) take_records<M>(a, sp.first + 1, sp.last, row, pre);      // while the last MMAs run
      if (mbar_wait_warp(&acc_full[2], 0)) {
        tc_fence_after();
        float acc[kNT];
        read_acc(tmem, quad, 2, nullptr, acc);
        if (sp.whole) {
          store_y<M>(a, yscale, tile_last, row, acc);
        } else if (fin) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (sp.first + 1 + i <= sp.last) {
#pragma unroll
              for (int m = 0; m < M; ++m) acc[m] += pre[i][m];
            }
          for (long long q = sp.first + 5; q <= sp.last; q += 4) {
            float v[4][M];
            take_records<M>(a, q, sp.last, row, v);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (q + i <= sp.last) {
#pragma unroll
                for (int m = 0; m < M; ++m) acc[m] += v[i][m];
              }
          }
          store_y<M>(a, yscale, tile_last, row, acc);
        } else {
          publish_record<M>(a, row, acc);
        }
      }
    }
  } else {
    // ---------------- epilogue: rows 32*quad .. 32*quad + 31 ----------------
    const int quad = warp & 3;
    griddep_wait();            // y and the records belong to the preceding kernel's era
    const float yscale = QX ? __fmul_rn(qg, __ldcg(a.wg)) : output_scale<BF>(a);
    // Every tile but the CTA's last (that one is flushed by the scale writers).
    const int tile_last = nunits > 0 ? (int)((u1 - 1) / C) : tile0 - 1;
    for (int tile = tile0, tile_idx = 0; tile < tile_last; ++tile, ++tile_idx) {
      const int d = tile_idx & 1;
      if (!mbar_wait_warp(&acc_full[d], (tile_idx >> 1) & 1)) break;
      tc_fence_after();
      float acc[kNT];
      read_acc(tmem, quad, d, &acc_empty[d], acc);
      // A tile before the last is whole, except the first when the range
      // starts inside it: then this CTA is not the tile's first contributor.
      if (tile == tile0 && u0 > (long long)tile0 * C) {
        publish_record<M>(a, quad * 32 + lane, acc);
      } else {
        store_y<M>(a, yscale, tile, quad * 32 + lane, acc);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <int S, bool QX = false>
constexpr size_t tc_smem_bytes() {
  return QX ? (size_t)S * kSlotQX + kResCodeBytes + kResScaleBytes + 1024 + (3 * S + 5 + kMaxRes) * sizeof(uint64_t) + 64
            : (size_t)S * kSlot + 1024 + (3 * S + 5) * sizeof(uint64_t) + 16;
}

struct TcMaps {
  CUtensorMap w_codes, w_scales, x_codes, x_scales;
};

// Test hook (nvfp4_test_gemv_fault): the record wait's poll limit and whether
// records are dropped, for every later launch in the process.
std::atomic<uint32_t> g_test_flag_spins{0};     // 0: kFlagSpinLimit
std::atomic<int> g_test_drop_records{0};

// Ring depth, read once per process (tuning knob NVFP4_GEMV_TC_STAGES: 4, 5 or 6).
int tc_stages() {
  static const int stages = [] {
    const char* st = getenv("NVFP4_GEMV_TC_STAGES");
    const int v = st ? atoi(st) : 4;
    return (v == 5 || v == 6) ? v : 4;
  }();
  return stages;
}

// CTAs of one instance that fit on an SM of the current device: shared memory
// (plus the 1 KB the driver reserves per CTA), TMEM columns and registers
// (allocated per warp in units of 256).  Sets the kernel's attributes on each
// device the first time; 0 and *err on failure.
template <int M, int S, bool BF, bool QX = false>
int tc_per_sm_fit(cudaError_t* err) {
  static PerDeviceInt fit;
  return fit.get([](int dev, cudaError_t* e_out) -> int {
    constexpr size_t smem = tc_smem_bytes<S, QX>();
    auto kern = gemv_tc_kernel<M, S, BF, QX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) {
      *e_out = e;
      return 0;
    }
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    const int by_smem = smem_sm > 0 ? (int)(smem_sm / (smem + 1024)) : 1;
    const int by_tmem = 512 / (int)kTmemCols;
    int by_regs = 2;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs > 0) {
      const int per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
      by_regs = 65536 / (per_warp * kWarps);
    }
    int f = by_smem < by_tmem ? by_smem : by_tmem;
    if (by_regs < f) f = by_regs;
    return f < 1 ? 1 : f;
  }, err);
}

}  // namespace

// Defined in gemv.cu.
bool nvfp4_internal_encode_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                              uint32_t box_inner, uint32_t box_rows, bool swizzle128);
int nvfp4_internal_device_sms();

// CTAs of the tensor-core GEMV per device (two per SM at the default depth).
static int tc_grid_max() { return 2 * nvfp4_internal_device_sms(); }

// Records: 128 x 8 words per CTA, at a fixed place in the workspace (they
// must stay zero between calls of any shape).
size_t nvfp4_internal_tc_record_bytes() { return (size_t)tc_grid_max() * kTR * 8 * sizeof(unsigned int); }

void nvfp4_internal_test_gemv_fault(unsigned int flag_spin_limit, int drop_records) {
  g_test_flag_spins.store(flag_spin_limit, std::memory_order_relaxed);
  g_test_drop_records.store(drop_records ? 1 : 0, std::memory_order_relaxed);
}
uint32_t nvfp4_internal_test_flag_spins() { return g_test_flag_spins.load(std::memory_order_relaxed); }
int nvfp4_internal_test_drop_records() { return g_test_drop_records.load(std::memory_order_relaxed); }

// The grid of an instance for a call (0 and *err on failure).
template <int M, int S, bool BF, bool QX>
static long long tc_grid(const TcArgs& a, int grid_cap, int max_ctas_per_sm, cudaError_t* err) {
  const int fit = tc_per_sm_fit<M, S, BF, QX>(err);
  if (fit == 0) return 0;
  const int per_sm = fit < max_ctas_per_sm ? fit : max_ctas_per_sm;
  long long G = (long long)per_sm * nvfp4_internal_device_sms();
  if (grid_cap > 0 && G > grid_cap) G = grid_cap;
  if (G > a.U) G = a.U;
  if (G > tc_grid_max()) G = tc_grid_max();  // records exist for that many CTAs
  return G;
}

// With the activation quantized in the kernel: whether every CTA's chunks fit
// its shared memory (kMaxRes) and its blocks stay within max_blocks.
static bool qx_fits(const TcArgs& a, long long G, long long max_blocks) {
  const long long most_units = (a.U + G - 1) / G;          // a CTA's units: floor or ceil of U / G
  const long long most_res = most_units < a.C ? most_units : a.C;
  return most_res <= kMaxRes && most_res * a.M * 16 <= max_blocks;
}

// Launches the kernel; with QX, only when qx_fits (*launched = false
// otherwise, nothing launched).
template <int M, int S, bool BF = false, bool QX = false>
static cudaError_t launch_tc(const TcMaps& mp, TcArgs a, cudaStream_t stream, int grid_cap, int max_ctas_per_sm,
                             bool* launched = nullptr, long long qx_max_blocks = 0) {
  cudaError_t e = cudaSuccess;
  if (launched) *launched = false;
  const long long G = tc_grid<M, S, BF, QX>(a, grid_cap, max_ctas_per_sm, &e);
  if (G == 0) return e;
  if (QX && !qx_fits(a, G, qx_max_blocks)) return cudaSuccess;
  const uint32_t spins = g_test_flag_spins.load(std::memory_order_relaxed);
  a.flag_spins = spins ? spins : kFlagSpinLimit;
  a.drop_records = g_test_drop_records.load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = tc_smem_bytes<S, QX>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel<M, S, BF, QX>, mp.w_codes, mp.w_scales, mp.x_codes, mp.x_scales, a);
  if (launched) *launched = true;
  return e;
}

template <int M>
static cudaError_t launch_tc_m(int stages, const TcMaps& mp, const TcArgs& a, cudaStream_t stream, int grid_cap,
                               int max_ctas_per_sm) {
  switch (stages) {
    case 5: return launch_tc<M, 5>(mp, a, stream, grid_cap, max_ctas_per_sm);
    case 6: return launch_tc<M, 6>(mp, a, stream, grid_cap, max_ctas_per_sm);
    default: return launch_tc<M, 4>(mp, a, stream, grid_cap, max_ctas_per_sm);
  }
}

// Tensor-core GEMV; the caller has validated the arguments.  Weights come either
// packed (wpacked != null, nvfp4_pack_weights layout) or as the row-major
// codes and scales wq, ws.  `records` holds nvfp4_internal_tc_record_bytes()
// bytes, zero between calls.
cudaError_t nvfp4_internal_gemv_tc(const uint8_t* xq, const uint8_t* xs, const float* xg, int M, const uint8_t* wq,
                                   const uint8_t* ws, const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                                   unsigned int* records, int grid_cap, int max_ctas_per_sm, cudaStream_t stream) {
  const int stages = tc_stages();
  TcMaps mp;
  memset(&mp, 0, sizeof(mp));   // the weight maps stay unused (and are never prefetched) for packed weights
  if (!wpacked && (!nvfp4_internal_encode_2d(&mp.w_codes, wq, (uint64_t)K / 2, (uint64_t)N, 128, kTR, true) ||
                   !nvfp4_internal_encode_2d(&mp.w_scales, ws, (uint64_t)K / 16, (uint64_t)N, 16, kTR, false)))
    return cudaErrorInvalidValue;
  if (!nvfp4_internal_encode_2d(&mp.x_codes, xq, (uint64_t)K / 2, (uint64_t)M, 128, kNT, true) ||
      !nvfp4_internal_encode_2d(&mp.x_scales, xs, (uint64_t)K / 16, (uint64_t)M, 16, kNT, false))
    return cudaErrorInvalidValue;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.wpacked = wpacked;
  a.xg = xg;
  a.wg = wg;
  a.y = y;
  a.records = records;
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = K / kChunk;
  a.RT = (N + kTR - 1) / kTR;
  a.U = (long long)a.RT * a.C;
  switch (M) {
    case 1: return launch_tc_m<1>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 2: return launch_tc_m<2>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 3: return launch_tc_m<3>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 4: return launch_tc_m<4>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 5: return launch_tc_m<5>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 6: return launch_tc_m<6>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    case 7: return launch_tc_m<7>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
    default: return launch_tc_m<8>(stages, mp, a, stream, grid_cap, max_ctas_per_sm);
  }
}

// Whether nvfp4_internal_quantize_gemv_tc would launch (the same grid and
// limits), without launching.
template <int M>
static cudaError_t qx_would_launch(const TcArgs& a, int grid_cap, int max_ctas_per_sm, long long max_blocks,
                                   bool* one) {
  cudaError_t e = cudaSuccess;
  const long long G = tc_grid<M, 4, false, true>(a, grid_cap, max_ctas_per_sm, &e);
  if (G == 0) return e;
  *one = qx_fits(a, G, max_blocks);
  return cudaSuccess;
}

cudaError_t nvfp4_internal_quantize_gemv_one_launch(int M, int N, int K, int grid_cap, int max_ctas_per_sm,
                                                    long long max_blocks, bool* one) {
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = K / kChunk;
  a.RT = (N + kTR - 1) / kTR;
  a.U = (long long)a.RT * a.C;
  *one = false;
  switch (M) {
    case 1: return qx_would_launch<1>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 2: return qx_would_launch<2>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 3: return qx_would_launch<3>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 4: return qx_would_launch<4>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 5: return qx_would_launch<5>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 6: return qx_would_launch<6>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    case 7: return qx_would_launch<7>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
    default: return qx_would_launch<8>(a, grid_cap, max_ctas_per_sm, max_blocks, one);
  }
}

// The activation quantizer and the GEMV in one launch (QX), packed weights,
// the default ring depth.  *launched = false when a CTA would hold more than
// kMaxRes activation chunks or quantize more than max_blocks blocks: the
// caller then quantizes and multiplies in two launches.
cudaError_t nvfp4_internal_quantize_gemv_tc(const uint16_t* x, int M, const uint8_t* wpacked, const float* wg, int N,
                                            int K, float* y, float* xg_out, unsigned int* records, int grid_cap,
                                            int max_ctas_per_sm, long long max_blocks, cudaStream_t stream,
                                            bool* launched) {
  TcMaps mp;
  memset(&mp, 0, sizeof(mp));   // no tensor maps: weights packed, activation quantized in the kernel
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.wpacked = wpacked;
  a.xg = nullptr;
  a.wg = wg;
  a.y = y;
  a.records = records;
  a.x = x;
  a.xg_out = xg_out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = K / kChunk;
  a.RT = (N + kTR - 1) / kTR;
  a.U = (long long)a.RT * a.C;
  switch (M) {
    case 1: return launch_tc<1, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 2: return launch_tc<2, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 3: return launch_tc<3, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 4: return launch_tc<4, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 5: return launch_tc<5, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 6: return launch_tc<6, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    case 7: return launch_tc<7, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
    default: return launch_tc<8, 4, false, true>(mp, a, stream, grid_cap, max_ctas_per_sm, launched, max_blocks);
  }
}

// BF16 y[M, N] = x[M, K] . w[N, K]^T on the same kernel (operands of kind::f16,
// no scales, units of [128 rows x 64 K]); the caller has validated the
// arguments (K a multiple of 64).
cudaError_t nvfp4_internal_bf16_gemv_tc(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                                        unsigned int* records, cudaStream_t stream) {
  TcMaps mp;
  memset(&mp, 0, sizeof(mp));   // no scale maps
  if (!nvfp4_internal_encode_2d(&mp.w_codes, w, (uint64_t)K * 2, (uint64_t)N, 128, kTR, true) ||
      !nvfp4_internal_encode_2d(&mp.x_codes, x, (uint64_t)K * 2, (uint64_t)M, 128, kNT, true))
    return cudaErrorInvalidValue;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.wpacked = nullptr;
  a.xg = nullptr;
  a.wg = nullptr;
  a.y = y;
  a.records = records;
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = K / 64;
  a.RT = (N + kTR - 1) / kTR;
  a.U = (long long)a.RT * a.C;
  switch (M) {
    case 1: return launch_tc<1, 4, true>(mp, a, stream, 0, 2);
    case 2: return launch_tc<2, 4, true>(mp, a, stream, 0, 2);
    case 3: return launch_tc<3, 4, true>(mp, a, stream, 0, 2);
    case 4: return launch_tc<4, 4, true>(mp, a, stream, 0, 2);
    case 5: return launch_tc<5, 4, true>(mp, a, stream, 0, 2);
    case 6: return launch_tc<6, 4, true>(mp, a, stream, 0, 2);
    case 7: return launch_tc<7, 4, true>(mp, a, stream, 0, 2);
    default: return launch_tc<8, 4, true>(mp, a, stream, 0, 2);
  }
}

// ---- weight packing -------------------------------------------------------------
namespace {
// One thread per 16-byte piece of the packed image: per block (tile t, chunk c)
// 1024 code pieces (row r, piece j stored at r*128 + ((j ^ (r & 7)) << 4)) and
// 128 scale pieces (row r at 16384 + 16 r); rows >= N are zero.
__global__ void __launch_bounds__(256) pack_weights_kernel(const uint8_t* __restrict__ wq,
                                                           const uint8_t* __restrict__ ws, int N, int K,
                                                           long long nblocks, uint8_t* __restrict__ packed) {
  constexpr int kPieces = kCodeBytes / 16 + kScaleBytes / 16;   // 1152
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblocks * kPieces) return;
  const long long blk = i / kPieces;
  const int p = (int)(i % kPieces);
  const int C = K / kChunk;
  const int t = (int)(blk / C), c = (int)(blk % C);
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  size_t dst = (size_t)blk * kPackedBlock;
  if (p < kCodeBytes / 16) {
    const int r = p >> 3, j = p & 7;
    const long long n = (long long)t * kTR + r;
    if (n < N) v = __ldg(reinterpret_cast<const uint4*>(wq + (size_t)n * (K / 2) + (size_t)c * 128 + j * 16));
    dst += (size_t)r * 128 + (size_t)((j ^ (r & 7)) << 4);
  } else {
    const int r = p - kCodeBytes / 16;
    const long long n = (long long)t * kTR + r;
    if (n < N) v = __ldg(reinterpret_cast<const uint4*>(ws + (size_t)n * (K / 16) + (size_t)c * 16));
    dst += (size_t)kCodeBytes + (size_t)r * 16;
  }
  *reinterpret_cast<uint4*>(packed + dst) = v;
}
}  // namespace

size_t nvfp4_internal_packed_bytes(int N, int K) {
  return (size_t)((N + kTR - 1) / kTR) * (size_t)(K / kChunk) * kPackedBlock;
}

cudaError_t nvfp4_internal_pack_weights(const uint8_t* wq, const uint8_t* ws, int N, int K, uint8_t* packed,
                                        cudaStream_t stream) {
  const long long nblocks = (long long)((N + kTR - 1) / kTR) * (K / kChunk);
  const long long pieces = nblocks * (kCodeBytes / 16 + kScaleBytes / 16);
  const long long grid = (pieces + 255) / 256;
  pack_weights_kernel<<<(unsigned)grid, 256, 0, stream>>>(wq, ws, N, K, nblocks, packed);
  return cudaGetLastError();
}
