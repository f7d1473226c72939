// Prefill-sized NVFP4 W4A4 GEMM on the tensor cores (tcgen05, sm_103a):
//   y[m, n] = xg * wg * sum_k e2m1(x[m,k]) e4m3(sx[m,k/16]) e2m1(w[n,k]) e4m3(sw[n,k/16]),  m < M <= 128.
//
// The pages measure their own tensor-core GEMM at M = 128 against vLLM's
// CUTLASS NVFP4 kernel (ReSET reading note §7.3, Table 16).  At M = 128 the
// product is still bound by the weight stream (2 * 128 flops per 0.5625 bytes
// of weights, about 455 flop/B, against a ridge near 2000 flop/B for FP4 on
// this GPU), so the kernel keeps the decode GEMV's plan -- each weight block
// read from HBM once, used for all tokens, Stream-K over [tile x 256-K]
// units with a deterministic fix-up -- and widens the token side of the MMA
// from 16 to 128:
//   tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X with
//   M = 128 weight rows (A, the packed weight block, one bulk copy) and
//   N = 128 tokens (B, a TMA tile of the row-major activation; rows >= M
//   arrive as zeros), K = 64 per instruction, 4 per 256-K stage.
// Block scales in TMEM (checked on sm_103a with an in-bounds probe): weight
// row r's 4 scales of an MMA at lane r, column A + r/32; token row n's at
// column B + n/32, lane 32p + n%32 of every lane quadrant p.  So per stage
// and MMA q: weight scales at columns SA + 4q + p, token scales at SB + 4q + g
// (g = n/32), 32 columns per stage.
//
// One CTA per SM (a ring of 6 stages of 36 KB: weight block + token tile);
// warps: 0 producer, 1 MMA issuer, 2-5 scale writers, 6-9 epilogue.  The
// 128-column FP32 accumulator is double buffered in TMEM; the epilogue reads
// it 16 token columns at a time.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "tcgen05.cuh"

NVFP4_DEFINE_ERROR_READER(nvfp4_internal_read_error_gemm)

namespace {

constexpr int kTR = 128;                    // weight rows per tile = MMA M
constexpr int kNT = 128;                    // MMA N: token rows (M <= 128 used, rest zero)
constexpr int kMaxTokens = 128;
constexpr int kChunk = 256;                 // K per stage
constexpr int kWCode = kTR * 128;           // 16384: weight codes, 128-byte rows, swizzled
constexpr int kWScale = kTR * 16;           // 2048
constexpr int kPackedBlock = kWCode + kWScale;
constexpr int kOffB = kPackedBlock;         // 18432 (1024-aligned): token codes, 128-byte rows, swizzled
constexpr int kOffSB = kOffB + kNT * 128;   // 34816: token scales, 16 bytes per row
constexpr int kSlot = kOffSB + kNT * 16;    // 36864 (36 x 1024)
constexpr uint32_t kStageTx = kSlot;        // every byte of a slot arrives by copy
constexpr int kStages = 6;
constexpr int kWarps = 10;
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kTmemCols = 512;         // D0 [0,128), D1 [128,256), 32 scale columns per stage from 256
constexpr uint32_t kColSF = 256;
static_assert(kColSF + 32 * kStages <= kTmemCols, "scale columns must fit the TMEM allocation");
// E2M1 x E2M1 (format 1), UE4M3 scales, K-major A and B, N = 128 (bits 17-22:
// N >> 3), M = 128 (bits 24-28: M >> 4), dense.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kNT >> 3) << 17) | ((uint32_t)(kTR >> 4) << 24);
constexpr uint32_t kFlagSpinLimit = 1u << 24;

struct GemmArgs {
  const uint8_t* wpacked;
  const float* xg;
  const float* wg;
  float* y;
  unsigned int* records;         // [G][M][128] words: a CTA's partial sums of its first tile; zero between calls
  int M, N, K, C;
  long long U;
  int tiles;                     // 128-row tiles: ceil(N / 128)
  int y_tma;                     // non-zero: a CTA's last tile goes out through shared memory and tm_y
  int cluster_k;                 // > 1: tile q / k of one CTA cluster of k, merged over distributed shared memory
  int whole_tiles;               // non-zero: CTA q takes tiles [q tiles / G, (q + 1) tiles / G) whole, no split
  uint32_t flag_spins;
  int drop_records;              // test hook (nvfp4_test_gemv_fault)
};

NVFP4_DEVINL unsigned int* record(const GemmArgs& a, long long q, int m, int row) {
  return a.records + ((size_t)q * a.M + m) * kTR + row;
}

// Reads accumulator columns [col, col + 16) of this warp's lane quadrant.
NVFP4_DEVINL void read16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Adds, in CTA order, the partial sums of contributors q0 .. q1 (at most
// kBatch of them) for tokens [m0, m0 + 16) of weight row `row` to v, once every
// word is written (bounded wait, device error bit 2 when it gives up); the live
// words are reset to zero.  All the batch's words are loaded in one pass, so a
// batch costs one L2 round trip when its records are in place.  A record word
// is the bitwise complement of an FP32 partial sum, so a written word is never
// zero.
constexpr int kBatch = 4;

NVFP4_DEVINL void take_batch(const GemmArgs& a, long long q0, long long q1, int m0, int row, float (&v)[16]) {
  unsigned int w[kBatch][16];
  // Every live word's load is issued before any is looked at (the loads are
  // ordered asm statements: a check between them would wait out each one's
  // L2 round trip in turn); only the words still zero are polled again.
#pragma unroll
  for (int j = 0; j < kBatch; ++j)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[j][i] = (q0 + j <= q1 && m0 + i < a.M) ? ld_relaxed_gpu(record(a, q0 + j, m0 + i, row)) : ~0u;
  uint32_t spins = 0;
  for (;;) {
    bool ready = true;
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
#pragma unroll
      for (int i = 0; i < 16; ++i) ready = ready && w[j][i] != 0u;
    if (ready) break;
    if (++spins >= a.flag_spins) {
      atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_FLAG_TIMEOUT);
      break;
    }
    __nanosleep(32);
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (w[j][i] == 0u) w[j][i] = ld_relaxed_gpu(record(a, q0 + j, m0 + i, row));
  }
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    if (q0 + j > q1) break;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] += __uint_as_float(~w[j][i]);
      if (m0 + i < a.M) st_relaxed_gpu(record(a, q0 + j, m0 + i, row), 0u);
    }
  }
}

// A CTA's last tile of y: the 128 x 128 FP32 block goes through the ring's
// shared memory (free by then: every unit's MMAs have completed) as two
// [128 tokens x 64 rows] boxes, written by two bulk tensor stores -- the tile's
// 64 KB in two copies instead of 128 scalar stores a thread.  Rows >= N and
// tokens >= M fall outside tm_y and are not written.
constexpr int kYBox = 64;                   // weight rows (FP32 columns of y) per store box: 256 bytes
constexpr int kMaxClusterK = 3;             // CTAs a tile in the cluster plan
NVFP4_DEVINL void tma_store_2d(const void* tmap, int32_t x, int32_t y, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(x),
               "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}

// Cluster-scope mbarrier operations and a distributed-shared-memory load, for
// the merge of a tile split across the CTAs of one cluster.
NVFP4_DEVINL void mbar_arrive_remote(uint64_t* local_bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(dsmem_addr(local_bar, rank))
               : "memory");
}
NVFP4_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMbarSpinLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_MBAR_TIMEOUT);
  return false;
}
NVFP4_DEVINL float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_xcodes,
                                                              const __grid_constant__ CUtensorMap tm_xscales,
                                                              const __grid_constant__ CUtensorMap tm_y,
                                                              const GemmArgs a) {
  constexpr int S = kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kSlot);
  uint64_t* sf_ready = full + S;
  uint64_t* empty = sf_ready + S;
  uint64_t* acc_full = empty + S;           // [0], [1]: alternating tiles
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* y_staged = acc_empty + 2;       // the 4 epilogue warps have staged the last tile
  uint64_t* part_ready = y_staged + 1;      // cluster rank 0: the other ranks' partial sums are staged
  uint64_t* consumed = part_ready + 1;      // other ranks: rank 0 has read this CTA's partial sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(consumed + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const int ck = a.cluster_k > 1 ? a.cluster_k : 1;
  const uint32_t crank = ck > 1 ? cluster_ctarank() : 0u;   // = blockIdx.x % ck: clusters are consecutive CTAs
  long long u0, u1;
  if (ck > 1) {                                  // one tile, its ck consecutive K ranges on the cluster's CTAs
    const long long t = blockIdx.x / ck;
    u0 = t * a.C + ((long long)crank * a.C) / ck;
    u1 = t * a.C + ((long long)(crank + 1) * a.C) / ck;
  } else if (a.whole_tiles) {
    u0 = ((long long)blockIdx.x * a.tiles / G) * a.C;
    u1 = ((long long)(blockIdx.x + 1) * a.tiles / G) * a.C;
  } else {
    u0 = unit_start(blockIdx.x, a.U, G);
    u1 = unit_start(blockIdx.x + 1, a.U, G);
  }
  const int nunits = (int)(u1 - u0);
  const int C = a.C;
  const int tile0 = (int)(u0 / C), chunk0 = (int)(u0 % C);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sf_ready[s], 4);
      mbar_init(&empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&acc_full[d], 1);
      mbar_init(&acc_empty[d], 4);
    }
    mbar_init(y_staged, 4);
    mbar_init(part_ready, 128 * (ck > 1 ? ck - 1 : 1));   // every epilogue thread of every other rank
    mbar_init(consumed, 128);                              // every epilogue thread of rank 0
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
  // A cluster's CTAs arrive once their barriers are initialised; a thread waits
  // before its first remote operation (the epilogue warps) or at the end.
  if (ck > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0 && nunits > 0) {
      prefetch_tmap(&tm_xcodes);
      prefetch_tmap(&tm_xscales);
      const int pre = nunits < S ? nunits : S;
      const uint8_t* wp = a.wpacked + (size_t)u0 * kPackedBlock;
      for (int k = 0; k < pre; ++k) {             // weights do not depend on the preceding kernel
        mbar_arrive_expect_tx(&full[k], kStageTx);
        bulk_g2s(smem + k * kSlot, wp + (size_t)k * kPackedBlock, kPackedBlock, &full[k]);
      }
      griddep_wait();                              // the tokens come from the preceding kernel
      int c = chunk0;
      for (int k = 0; k < pre; ++k) {
        uint8_t* slot = smem + k * kSlot;
        tma_load_2d(slot + kOffB, &tm_xcodes, c * 128, 0, &full[k]);
        tma_load_2d(slot + kOffSB, &tm_xscales, c * 16, 0, &full[k]);
        if (++c == C) c = 0;
      }
      int issued = pre;
      int s = pre % S;
      uint32_t phase = (pre / S) & 1;
      for (int k = pre; k < nunits; ++k) {
        if (!mbar_wait(&empty[s], phase ^ 1u)) break;
        uint8_t* slot = smem + s * kSlot;
        mbar_arrive_expect_tx(&full[s], kStageTx);
        bulk_g2s(slot, wp + (size_t)k * kPackedBlock, kPackedBlock, &full[s]);
        tma_load_2d(slot + kOffB, &tm_xcodes, c * 128, 0, &full[s]);
        tma_load_2d(slot + kOffSB, &tm_xscales, c * 16, 0, &full[s]);
        issued = k + 1;
        if (++c == C) c = 0;
        if (++s == S) { s = 0; phase ^= 1u; }
      }
      for (int k = (issued > S ? issued - S : 0); k < issued; ++k) mbar_wait(&full[k % S], (k / S) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread) ----------------
    // The loop is unrolled by ring stage, so each unit's descriptors and scale
    // columns are compile-time offsets from the stage-0 values: this thread
    // is the unit loop's limit (an MMA issue holds it, and every instruction
    // between the MMAs adds to the unit), so it does as little as it can.
    if (lane == 0 && nunits > 0) {
      const uint64_t da0 = smem_desc_sw128(smem_u32(smem));
      const uint64_t db0 = smem_desc_sw128(smem_u32(smem + kOffB));
      const uint32_t sf0 = tmem + kColSF;
      int tile_idx = 0;
      int left = C - chunk0;                // units left in the current tile
      bool first = true;                    // the next unit starts a tile
      uint32_t phase = 0;
      int issued = 0;
      uint32_t d_tmem = tmem;
      bool ok = true;
      while (ok && issued < nunits) {
#pragma unroll
        for (int st = 0; st < S; ++st) {
          if (issued == nunits) break;
          if (first) {
            if (tile_idx >= 2 && !mbar_wait(&acc_empty[tile_idx & 1], ((tile_idx >> 1) - 1) & 1)) {
              ok = false;
              break;
            }
            d_tmem = tmem + (uint32_t)((tile_idx & 1) * kNT);
          }
          if (!mbar_wait(&sf_ready[st], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t doff = (uint64_t)((st * kSlot) >> 4);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            mma_mxf4nvf4(d_tmem, da0 + doff + 2 * q, db0 + doff + 2 * q, kIdesc, sf0 + 32u * st + 4u * q,
                         sf0 + 32u * st + 16u + 4u * q, (first && q == 0) ? 0u : 1u);
          mma_commit(&empty[st]);
          ++issued;
          first = false;
          if (--left == 0 || issued == nunits) {        // last unit of this tile
            mma_commit(&acc_full[tile_idx & 1]);
            ++tile_idx;
            left = C;
            first = true;
          }
        }
        phase ^= 1u;
      }
      if (issued > 0) mbar_wait(&empty[(issued - 1) % S], ((issued - 1) / S) & 1);
    }
  } else if (warp < 6) {
    // ---------------- scale writers: this warp's lane quadrant p ----------------
    const int p = warp & 3;
    const uint32_t qbase = tmem + ((uint32_t)(p * 32) << 16) + kColSF;
    int s = 0;
    uint32_t phase = 0;
    for (int k = 0; k < nunits; ++k) {
      if (!mbar_wait_warp(&full[s], phase)) break;
      const uint8_t* slot = smem + s * kSlot;
      const uint32_t col = qbase + 32u * s;
      // weight row 32p + lane: its 4 words (one per MMA q) at columns 4q + p
      const uint4 sa = *reinterpret_cast<const uint4*>(slot + kOffB - kWScale + (p * 32 + lane) * 16);
      tmem_st1(col + (uint32_t)p, sa.x);
      tmem_st1(col + 4u + (uint32_t)p, sa.y);
      tmem_st1(col + 8u + (uint32_t)p, sa.z);
      tmem_st1(col + 12u + (uint32_t)p, sa.w);
      // token row 32g + lane: its 4 words at columns 16 + 4q + g, in every quadrant
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 sb = *reinterpret_cast<const uint4*>(slot + kOffSB + (g * 32 + lane) * 16);
        tmem_st1(col + 16u + (uint32_t)g, sb.x);
        tmem_st1(col + 20u + (uint32_t)g, sb.y);
        tmem_st1(col + 24u + (uint32_t)g, sb.z);
        tmem_st1(col + 28u + (uint32_t)g, sb.w);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_ready[s]);
      if (++s == S) { s = 0; phase ^= 1u; }
    }
  } else {
    // ---------------- epilogue: weight rows 32p .. 32p + 31 ----------------
    const int p = warp & 3;
    const int row = p * 32 + lane;
    griddep_wait();            // y and the records belong to the preceding kernel's era
    if (ck > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    const float yscale = __fmul_rn(__ldcg(a.xg), __ldcg(a.wg));
    const int tile_last = nunits > 0 ? (int)((u1 - 1) / C) : tile0 - 1;
    for (int tile = tile0, tile_idx = 0; tile <= tile_last; ++tile, ++tile_idx) {
      const int d = tile_idx & 1;
      if (!mbar_wait_warp(&acc_full[d], (tile_idx >> 1) & 1)) break;
      tc_fence_after();
      // Split tiles: a cluster's ranks 1..k-1 stage their partial sums in their
      // own shared memory and rank 0 adds them; otherwise the tile's first CTA
      // adds the others' records (Stream-K).
      const bool cl = ck > 1;
      const bool partner = cl && crank != 0;
      bool whole, fin;
      long long first = 0, last = 0;
      if (cl) {
        whole = false;
        fin = crank == 0;
      } else {
        const long long t0 = (long long)tile * C;
        first = cta_of_unit(t0, a.U, G);
        last = cta_of_unit(t0 + C - 1, a.U, G);
        whole = a.whole_tiles || first == last;
        fin = !whole && first == (long long)blockIdx.x;   // this CTA finishes the split tile
      }
      const int n = tile * kTR + row;
      const uint32_t dcol = tmem + ((uint32_t)(p * 32) << 16) + (uint32_t)(d * kNT);
      const bool staged = a.y_tma && tile == tile_last && (whole || fin);
      // box (row / 64): [token m][row % 64] floats, 256 bytes a token -- the
      // staging of y, and of a cluster rank's partial sums
      float* stage = reinterpret_cast<float*>(smem + (row / kYBox) * (kNT * kYBox * 4)) + (row % kYBox);
      if (fin && cl) {
        // Rank 0: every thread acquires the partials, then adds the other ranks'
        // values of its row in rank order, the next 16 tokens' loads issued
        // before the current ones are added (a load's round trip is long).
        if (!mbar_wait_cluster(part_ready, 0)) break;
        float wq[kMaxClusterK - 1][16];
#pragma unroll
        for (int r = 1; r < kMaxClusterK; ++r)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            wq[r - 1][i] = r < ck ? ld_dsmem_f32(dsmem_addr(&stage[i * kYBox], (uint32_t)r)) : 0.0f;
        for (int m0 = 0; m0 < a.M; m0 += 16) {
          float v[16];
          read16(dcol + (uint32_t)m0, v);
          float wn[kMaxClusterK - 1][16];
          const bool more = m0 + 16 < a.M;
#pragma unroll
          for (int r = 1; r < kMaxClusterK; ++r)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              wn[r - 1][i] = (more && r < ck) ? ld_dsmem_f32(dsmem_addr(&stage[(m0 + 16 + i) * kYBox], (uint32_t)r)) : 0.0f;
#pragma unroll
          for (int r = 1; r < kMaxClusterK; ++r)
            if (r < ck) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] += wq[r - 1][i];
            }
          if (staged) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stage[(m0 + i) * kYBox] = v[i] * yscale;
          } else if (n < a.N) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (m0 + i < a.M) a.y[(size_t)(m0 + i) * a.N + n] = v[i] * yscale;
          }
#pragma unroll
          for (int r = 0; r < kMaxClusterK - 1; ++r)
#pragma unroll
            for (int i = 0; i < 16; ++i) wq[r][i] = wn[r][i];
        }
      } else
      for (int m0 = 0; m0 < a.M; m0 += 16) {
        float v[16];
        read16(dcol + (uint32_t)m0, v);
        if (partner) {
#pragma unroll
          for (int i = 0; i < 16; ++i) stage[(m0 + i) * kYBox] = v[i];
        } else if (whole || fin) {
          if (fin) {                  // in CTA order: a fixed order of additions
            for (long long q = first + 1; q <= last; q += kBatch)
              take_batch(a, q, q + kBatch - 1 < last ? q + kBatch - 1 : last, m0, row, v);
          }
          if (staged) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stage[(m0 + i) * kYBox] = v[i] * yscale;
          } else if (n < a.N) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (m0 + i < a.M) a.y[(size_t)(m0 + i) * a.N + n] = v[i] * yscale;
          }
        } else if (!a.drop_records) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (m0 + i < a.M) st_relaxed_gpu(record(a, blockIdx.x, m0 + i, row), ~__float_as_uint(v[i]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[d]);
      if (partner) {
        // This thread's partial sums are staged: tell rank 0, then keep the
        // shared memory until rank 0 has read it (bounded wait).
        mbar_arrive_remote(part_ready, 0u);
        if (p == 2 && lane == 0) mbar_wait_cluster(consumed, 0);
      } else if (fin && cl) {
        // this thread has read its rows of every other rank's partial sums
        for (int r = 1; r < ck; ++r) mbar_arrive_remote(consumed, (uint32_t)r);
      }
      if (staged) {
        // Each warp makes its writes visible to the copy engine and arrives; one
        // thread waits (bounded) for the four, then issues the copies and waits
        // for them.  The other threads do not wait.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(y_staged);
        if (p == 2 && lane == 0 && mbar_wait(y_staged, 0)) {
          for (int b = 0; b < kTR / kYBox; ++b)
            tma_store_2d(&tm_y, (tile * kTR + b * kYBox) * 4, 0, smem + b * (kNT * kYBox * 4));
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
      }
    }
  }
  tc_fence_before();
  if (ck > 1 && warp < 6) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // (epilogue warps: above)
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

constexpr size_t gemm_smem_bytes() { return (size_t)kStages * kSlot + 1024 + (3 * kStages + 7) * sizeof(uint64_t) + 16; }

}  // namespace

// Defined in gemv.cu.
bool nvfp4_internal_encode_2d(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                              uint32_t box_inner, uint32_t box_rows, bool swizzle128);
int nvfp4_internal_device_sms();
// Defined in gemv_tc.cu: the test hook's settings.
uint32_t nvfp4_internal_test_flag_spins();
int nvfp4_internal_test_drop_records();

// Records: 128 tokens x 128 rows of words per CTA, one CTA per SM.
size_t nvfp4_internal_gemm_record_bytes() {
  return (size_t)nvfp4_internal_device_sms() * kMaxTokens * kTR * sizeof(unsigned int);
}

// The caller has validated the arguments (M 1..128, K a multiple of 256,
// packed weights); `records` holds nvfp4_internal_gemm_record_bytes() bytes,
// zero between calls.
cudaError_t nvfp4_internal_gemm_tc(const uint8_t* xq, const uint8_t* xs, const float* xg, int M, const uint8_t* wpacked,
                                   const float* wg, int N, int K, float* y, unsigned int* records,
                                   cudaStream_t stream) {
  static PerDeviceInt attr_set;
  cudaError_t err = cudaSuccess;
  if (attr_set.get([](int, cudaError_t* e_out) -> int {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gemm_smem_bytes());
        if (e != cudaSuccess) {
          *e_out = e;
          return 0;
        }
        return 1;
      }, &err) == 0)
    return err;
  CUtensorMap mx, ms;
  if (!nvfp4_internal_encode_2d(&mx, xq, (uint64_t)K / 2, (uint64_t)M, 128, kNT, true) ||
      !nvfp4_internal_encode_2d(&ms, xs, (uint64_t)K / 16, (uint64_t)M, 16, kNT, false))
    return cudaErrorInvalidValue;
  GemmArgs a;
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
  a.U = (long long)((N + kTR - 1) / kTR) * a.C;
  const uint32_t spins = nvfp4_internal_test_flag_spins();
  a.flag_spins = spins ? spins : kFlagSpinLimit;
  a.drop_records = nvfp4_internal_test_drop_records();
  // One CTA per SM, in one of two plans, whichever leaves the busiest CTA the
  // less work in units of one [128-row x 256-K] MMA step:
  //  - whole tiles: CTA q takes tiles [q T / G, (q + 1) T / G), at most
  //    ceil(T / SMs) of them; nothing to merge;
  //  - split tiles: with fewer tiles than SMs every tile gets the same whole
  //    number of CTAs (T x floor(SMs / T)), else Stream-K over all SMs; a split
  //    tile's finishing CTA then merges 64 KB of partial sums per contributor
  //    at M = 128, which measured as long as about 4.5 MMA steps per 16 tokens.
  // (Qwen3-32B at M = 128: whole tiles for qkv and gate_up; clusters of two
  // for o and of three for down, whose 40 tiles would leave 112 SMs idle.)
  const long long sms = nvfp4_internal_device_sms();
  const long long tiles = (N + kTR - 1) / kTR;
  a.tiles = (int)tiles;
  const long long per = (tiles + sms - 1) / sms;
  const long long g_whole = (tiles + per - 1) / per;
  long long g_split = tiles < sms ? tiles * (sms / tiles) : sms;
  if (g_split > a.U) g_split = a.U;
  const bool splits = !(g_split <= tiles && tiles % g_split == 0);
  const long long cost_whole = per * a.C;
  const long long cost_split = (a.U + g_split - 1) / g_split + (splits ? (9 * ((M + 15) / 16) + 1) / 2 : 0);
  // With fewer tiles than SMs, a tile can also go to a cluster of k <= 3 CTAs
  // (k <= units a tile) whose partial sums meet in shared memory: each other
  // rank stages 64 KB at M = 128, rank 0 reads it over distributed shared
  // memory and adds it -- about 1.5 MMA steps per 16 tokens per rank, as
  // fitted to whole calls at M = 128 (time = fixed + steps x 0.25 us: o on
  // two ranks and down on three both gave 1.5-1.6).  Ties go to the larger
  // cluster.
  long long best_k = 1, cost_cluster = -1;
  for (long long k = 2; k <= kMaxClusterK && tiles * k <= sms && k <= a.C; ++k) {
    const long long c = (a.C + k - 1) / k + (k - 1) * 3 * ((M + 15) / 16) / 2;
    if (cost_cluster < 0 || c <= cost_cluster) {
      cost_cluster = c;
      best_k = k;
    }
  }
  static const int mode = [] {            // tuning knob NVFP4_GEMM_MODE: "tiles", "split" or "cluster" forces a plan
    const char* v = getenv("NVFP4_GEMM_MODE");
    return (v && v[0] == 't') ? 1 : (v && v[0] == 's') ? 2 : (v && v[0] == 'c') ? 3 : 0;
  }();
  int plan;                               // 1 whole tiles, 2 split tiles, 3 cluster
  if (mode == 1 || mode == 2) {
    plan = mode;
  } else if (mode == 3) {
    plan = best_k > 1 ? 3 : 1;
  } else {
    plan = cost_whole <= cost_split ? 1 : 2;
    if (best_k > 1 && cost_cluster < (plan == 1 ? cost_whole : cost_split)) plan = 3;
  }
  long long G = plan == 1 ? g_whole : plan == 2 ? g_split : tiles * best_k;
  a.whole_tiles = plan == 1 ? 1 : 0;
  a.cluster_k = plan == 3 ? (int)best_k : 1;
  if (G > a.U) G = a.U;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)a.cluster_k;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster_k > 1 ? 2 : 1;
  // y through bulk tensor stores when its rows are 16-byte multiples (N % 4 == 0)
  // on a 16-byte aligned base; else plain stores (tm_y unused).
  CUtensorMap my;
  memset(&my, 0, sizeof(my));
  a.y_tma = (N % 4 == 0) && nvfp4_internal_encode_2d(&my, y, (uint64_t)N * 4, (uint64_t)M, kYBox * 4, kNT, false);
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, mx, ms, my, a);
}

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);
nvfp4_status nvfp4_internal_check_device();

extern "C" size_t nvfp4_gemm_workspace_bytes(int M, int N, int K) {
  if (M < 1 || M > kMaxTokens || N < 1 || N > (1 << 20) || K < kChunk || (K % kChunk) != 0) return 0;
  return (nvfp4_internal_gemm_record_bytes() + 255) & ~(size_t)255;
}

extern "C" nvfp4_status nvfp4_gemm_packed(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                          const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!xq || !xs || !xg || !wpacked || !wg || !y || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxTokens) return NVFP4_ERR_RANGE;
  if (N < 1 || N > (1 << 20) || K < kChunk || (K % kChunk) != 0) return NVFP4_ERR_SHAPE;
  if (!nvfp4_internal_aligned(xq, 16) || !nvfp4_internal_aligned(xs, 16) || !nvfp4_internal_aligned(wpacked, 16) ||
      !nvfp4_internal_aligned(y, 16) || !nvfp4_internal_aligned(xg, 4) || !nvfp4_internal_aligned(wg, 4) ||
      !nvfp4_internal_aligned(workspace, 256))
    return NVFP4_ERR_ALIGN;
  if (workspace_bytes < nvfp4_gemm_workspace_bytes(M, N, K)) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  return nvfp4_internal_cuda_status(nvfp4_internal_gemm_tc(xq, xs, xg, M, wpacked, wg, N, K, y,
                                                           static_cast<unsigned int*>(workspace), stream));
}
