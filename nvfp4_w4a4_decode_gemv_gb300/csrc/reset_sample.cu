// ReSET step-aware temperature sampler (one decode position, M rows).
//
// Rule (ReSET project page, "Step-aware temperature scaling"; reading note
// §3.1 Eq. (1), §3.2, §4.1 SAT, §4.2 HSE, §4.3):
//   H      = entropy of softmax(logits)            (nats, temperature 1)
//   H_step = mean of the last w entropies while the in-step position j < w,
//            else the running mean of the step's entropies
//   H_bar  = running mean of all entropies of the sequence
//   tau    = tau0 if H_step <= H_bar (confident step) else H_step
//            (or, for the two policies ReSET is compared against -- reading
//            note §3.1 Eq. (1) and §6.3 Table 2 -- tau0 always, or the mean
//            of the last w entropies)
//   T      = T_low if H < tau else T_high
//   token  = min{ i : sum_{k<=i} p_k > u * sum_k p_k },  p_k = exp((l_k - max l) / T)
//            over the top-p nucleus when top_p is set (reading note §6.1)
//
// One launch: grid = M rows x NC chunks of kChunk logits.  Each CTA reduces its
// chunk to (max m, the number of logits equal to m, sum of e^(l-m) over the
// others, sum e^(l-m)(l-m), sum e^((l-m)/T_low), sum e^((l-m)/T_high)) in FP32
// and publishes it (keeping the terms equal to 1 out of the FP32 sum keeps the
// small tail of a peaked distribution, and so its entropy, accurate); the last CTA of a row to
// arrive (atomic counter, no spin-wait) merges the chunks in chunk order in
// FP64 -- deterministic whichever CTA is last -- updates the row's state,
// picks T, finds the chunk that holds u * Z_T and scans that one chunk with an
// FP64 prefix sum.  It resets the row counter for the next call.
//
// With top-p, the last CTA stops after choosing T and four more launches of
// M x NC CTAs follow: three levels of a radix select over the logits' order
// keys (11, 11 and 10 bits) that find the least probable kept logit, and one
// that sums each chunk's kept mass and samples.  Masses there are integers
// (exp((l - max) / T) scaled by 2^(62 - ceil(log2 V)) and rounded), so every
// level, the chunk sums and the final scan see the same numbers and the sums
// are exact in any order: the result is deterministic, and the per-row
// histograms can be accumulated with atomics.
#include <math.h>

#include <mutex>

#include "common.cuh"

NVFP4_DEFINE_ERROR_READER(nvfp4_internal_read_error_reset)

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;
constexpr int kChunk = kThreads * kPerThread;     // 2048 logits per CTA
constexpr int kMaxRows = 64;
constexpr int kMaxW = 256;

struct RowState {           // per-row state, followed by `w` doubles (the entropy ring)
  int t;                    // positions seen
  int j;                    // 0-based position inside the current step
  int w;
  int pad;
  double glob_sum;          // sum of all entropies
  double step_sum;          // sum of the current step's entropies
};

struct Params {
  float tau0, t_low, t_high;
  int w;
  int threshold;            // RESET_THRESHOLD_*
  float top_p;              // in (0, 1): sample from the nucleus, else from every token
  float mscale;             // integer-mass scale of the nucleus: 2^(62 - ceil(log2 V))
};

constexpr int kHistBins = 2048;   // per-row histogram of one radix level

// Per-row record of the top-p launches.
struct NucRow {
  float gmax, T;                   // row maximum and chosen temperature (first launch)
  unsigned int prefix;             // key bits chosen so far; the boundary key after level 2
  unsigned int pad;
  unsigned long long below;        // kept mass of the keys before the current prefix's range
  unsigned long long target;       // ceil(top_p * Z), Z the row's total integer mass
  unsigned long long zk;           // the nucleus's integer mass
  unsigned long long pad2[3];
};

// Order key of a logit: ascending as the logit falls, equal for equal logits
// (-0 and +0 included).
__device__ __forceinline__ uint32_t nucleus_key(float l) {
  uint32_t b = __float_as_uint(l);
  if (b == 0x80000000u) b = 0u;
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);   // ascending with l
  return ~ord;
}

// Integer mass of a logit at temperature 1/invT, relative to the row maximum.
__device__ __forceinline__ unsigned long long nucleus_mass(float l, float gmax, float invT, float mscale) {
  return __float2ull_rn(expf((l - gmax) * invT) * mscale);
}

size_t state_stride(int w) { return (sizeof(RowState) + (size_t)w * sizeof(double) + 15) & ~size_t(15); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per-chunk partials, padded to 8 floats.
struct Part {
  float mx, z1, a1, zl, zh, n0, pad0, pad1;   // z1, a1 exclude the n0 logits equal to mx
};

__global__ void __launch_bounds__(kThreads) reset_sample_kernel(const float* __restrict__ logits, int M, int V, int NC,
                                                               const uint8_t* __restrict__ step_start,
                                                               const float* __restrict__ u, uint8_t* state,
                                                               int stride, Params p, int32_t* token, float* H_out,
                                                               float* T_out, Part* parts, unsigned int* counters,
                                                               NucRow* nrows, unsigned long long* hist) {
  __shared__ float s_red[5][kThreads / 32];
  __shared__ int s_last;
  __shared__ double s_scan[kThreads / 32];
  __shared__ double s_zt[1024];          // per-chunk Z_T (rescaled to the row max); NC <= 1024
  __shared__ double s_target;
  __shared__ float s_T, s_rowmax;
  __shared__ int s_chunk;
  __shared__ int s_tok;

  const int row = blockIdx.x / NC, c = blockIdx.x % NC;
  const float* base = logits + (size_t)row * V;
  const int lo = c * kChunk;
  const int hi = min(V, lo + kChunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- chunk partials ----
  float v[kPerThread];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int i = lo + threadIdx.x + k * kThreads;
    v[k] = (i < hi) ? __ldg(base + i) : -INFINITY;
    mx = fmaxf(mx, v[k]);
  }
  mx = warp_max(mx);
  if (lane == 0) s_red[0][warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int w = 0; w < kThreads / 32; ++w) m = fmaxf(m, s_red[0][w]);
    s_rowmax = m;
  }
  __syncthreads();
  const float cm = s_rowmax;
  const float inv_tl = 1.0f / p.t_low, inv_th = 1.0f / p.t_high;   // same expressions as below
  float n0 = 0.f, z1 = 0.f, a1 = 0.f, zl = 0.f, zh = 0.f;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int i = lo + threadIdx.x + k * kThreads;
    if (i < hi) {
      const float s = v[k] - cm;
      if (s == 0.0f) {
        n0 += 1.0f;                      // e^0 = 1, counted exactly
      } else {
        const float e = expf(s);
        z1 += e;
        if (e > 0.0f) a1 += e * s;       // a -inf logit adds nothing (not 0 x -inf)
      }
      zl += expf(s * inv_tl);
      zh += expf(s * inv_th);
    }
  }
  n0 = warp_sum(n0);
  z1 = warp_sum(z1);
  a1 = warp_sum(a1);
  zl = warp_sum(zl);
  zh = warp_sum(zh);
  __syncthreads();
  if (lane == 0) {
    s_red[0][warp] = z1;
    s_red[1][warp] = a1;
    s_red[2][warp] = zl;
    s_red[3][warp] = zh;
    s_red[4][warp] = n0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Part q;
    q.mx = cm;
    q.z1 = q.a1 = q.zl = q.zh = q.n0 = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) {
      q.z1 += s_red[0][w];
      q.a1 += s_red[1][w];
      q.zl += s_red[2][w];
      q.zh += s_red[3][w];
      q.n0 += s_red[4][w];
    }
    __stcg(reinterpret_cast<float4*>(parts + (size_t)row * NC + c), make_float4(q.mx, q.z1, q.a1, q.zl));
    __stcg(reinterpret_cast<float4*>(parts + (size_t)row * NC + c) + 1, make_float4(q.zh, q.n0, 0.f, 0.f));
    __threadfence();
    s_last = (atomicAdd(counters + row, 1u) == (unsigned int)(NC - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of the row: merge chunk partials in chunk order (FP64) ----
  if (warp == 0) {
    // Each lane's first kCached chunk partials are loaded together and kept in
    // registers for both passes (one round of L2 latency instead of one per
    // chunk and pass); chunks beyond 32 * kCached (V > 262144) are reloaded.
    constexpr int kCached = 4;
    const float4* prow = reinterpret_cast<const float4*>(parts + (size_t)row * NC);
    float4 c0[kCached], c1[kCached];
#pragma unroll
    for (int i = 0; i < kCached; ++i) {
      const int q = lane + 32 * i;
      c0[i] = q < NC ? __ldcg(prow + 2 * q) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
      c1[i] = q < NC ? __ldcg(prow + 2 * q + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float gmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCached; ++i) gmax = fmaxf(gmax, c0[i].x);
    for (int q = lane + 32 * kCached; q < NC; q += 32) gmax = fmaxf(gmax, __ldcg(&parts[(size_t)row * NC + q].mx));
    gmax = warp_max(gmax);
    double Z = 0.0, A = 0.0;
    auto add = [&](const float4& p0, const float4& p1) {
      const float d = p0.x - gmax;                      // <= 0
      const double r1 = (double)expf(d);
      Z += r1 * ((double)p1.y + (double)p0.y);
      A += r1 * ((double)p0.z + (double)d * ((double)p0.y + (double)p1.y));
    };
#pragma unroll
    for (int i = 0; i < kCached; ++i)
      if (lane + 32 * i < NC) add(c0[i], c1[i]);
    for (int q = lane + 32 * kCached; q < NC; q += 32) add(__ldcg(prow + 2 * q), __ldcg(prow + 2 * q + 1));
    Z = warp_sum_d(Z);
    A = warp_sum_d(A);
    if (lane == 0) {
      // The logarithm and the mean in FP32: FP64 is a narrow pipe on this part
      // and this chain is serial.  Z >= 1 (the maximum contributes e^0), and
      // Z - 1 is formed in FP64 so that log1p keeps its relative precision
      // when the distribution is nearly one-hot (H -> 0); the two terms have
      // the same sign, so H keeps ~1e-7 relative error against a 1e-4
      // tolerance.
      const double H = (double)(log1pf((float)(Z - 1.0)) - (float)A / (float)Z);
      // ---- ReSET state update (FP64 sums) ----
      RowState* st = reinterpret_cast<RowState*>(state + (size_t)row * stride);
      double* ring = reinterpret_cast<double*>(st + 1);
      // The ring holds st->w entries; a call with another window than the one
      // the state was initialised with is an error: recorded, and the row is
      // sampled at T_high without touching its state.
      const int w = p.w;
      const bool state_ok = (st->w == w);
      if (!state_ok) atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_STATE_W);
      double Hs = 0.0, Hbar = 0.0, Hwin = 0.0;
      int t1 = 0, j = 0;
      if (state_ok) {
        if (st->t == 0 || (step_start && step_start[row])) {
          st->j = 0;
          st->step_sum = 0.0;
        }
        st->glob_sum += H;
        st->step_sum += H;
        ring[st->t % w] = H;
        t1 = st->t + 1;
        j = st->j;
        if (t1 <= w) {
          Hwin = st->glob_sum / t1;             // the window is the whole history
        } else {
          double ws = 0.0;
          for (int i = 0; i < w; ++i) ws += ring[i];
          Hwin = ws / w;
        }
        Hs = (j < w) ? Hwin : st->step_sum / (j + 1);
        Hbar = st->glob_sum / t1;
      }
      const double tau = (p.threshold == RESET_THRESHOLD_FIXED)    ? (double)p.tau0
                         : (p.threshold == RESET_THRESHOLD_WINDOW) ? Hwin
                         : (Hs <= Hbar)                            ? (double)p.tau0
                                                                   : Hs;
      const bool low = state_ok && H < tau;
      const float T = low ? p.t_low : p.t_high;
      if (state_ok) {
        st->t = t1;
        st->j = j + 1;
      }
      if (H_out) H_out[row] = (float)H;
      if (T_out) T_out[row] = T;
      s_T = T;
      s_rowmax = gmax;
      s_target = (double)__ldg(u + row);      // scaled by Z_T below
    }
  }
  __syncthreads();
  const float T = s_T, gmax = s_rowmax;
  if (nrows) {
    // top-p: hand the row over to the nucleus launches; clear its histogram.
    unsigned long long* h = hist + (size_t)row * kHistBins;
    for (int b = threadIdx.x; b < kHistBins; b += kThreads) h[b] = 0ull;
    if (threadIdx.x == 0) {
      NucRow nr = {};
      nr.gmax = gmax;
      nr.T = T;
      nrows[row] = nr;
      counters[row] = 0u;
    }
    return;
  }
  const float invT = 1.0f / T;
  const bool use_low = (T == p.t_low);
  // per-chunk Z_T rescaled to the row max, then the chunk that holds the target
  for (int q = threadIdx.x; q < NC; q += kThreads) {
    const float4 p0 = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)row * NC + q));
    const float4 p1 = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)row * NC + q) + 1);
    s_zt[q] = (double)expf((p0.x - gmax) * invT) * (double)(use_low ? p0.w : p1.x);
  }
  __syncthreads();
  if (warp == 0) {
    // The first chunk whose cumulative Z_T passes the target (the last chunk
    // if rounding leaves the target at or past the total).  Lane L owns the
    // consecutive chunks [L per, (L+1) per): per-lane sums, an inclusive scan
    // across the warp, and the first lane whose running sum passes the target
    // walks its own chunks (a serial loop over all chunks cost 6 us in FP64).
    const int per = (NC + 31) / 32;
    const int q0 = lane * per, q1 = min(NC, q0 + per);
    double mine = 0.0;
    for (int q = q0; q < q1; ++q) mine += s_zt[q];
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const double total = __shfl_sync(0xffffffffu, incl, 31);
    const double target = s_target * total;     // s_target holds u until here
    const unsigned hit = __ballot_sync(0xffffffffu, q0 < q1 && incl > target);
    const int owner = hit ? __ffs(hit) - 1 : (NC - 1) / per;
    if (lane == owner) {
      // The owner's last chunk is the fallback: the walk re-adds in its own
      // order, so it may stop short of a target that `incl` passed by a
      // rounding; for the last lane this is the "last chunk" case.
      double before = incl - mine;
      int cstar = q1 - 1;
      for (int q = q0; q < q1 - 1; ++q) {
        if (before + s_zt[q] > target) {
          cstar = q;
          break;
        }
        before += s_zt[q];
      }
      s_chunk = cstar;
      s_target = target - before;
      s_tok = 0x7fffffff;
    }
  }
  __syncthreads();
  // ---- scan the chosen chunk: thread t owns 8 consecutive logits ----
  const int clo = s_chunk * kChunk;
  const int chi = min(V, clo + kChunk);
  // The thread's 8 running sums in FP32 (relative error <= 8 roundings of the
  // thread's sum, far inside the 4e-6 Z tolerance of the sample); the scan
  // across threads and the comparisons in FP64.
  float pre[kPerThread];
  float fsum = 0.0f;
  {
    const int i0 = clo + threadIdx.x * kPerThread;
    float lv[kPerThread];
    // 16-byte loads only where the row start is 16-byte aligned (V a multiple
    // of 4; logits itself is checked 16-byte aligned) and all 8 are in range.
    if ((V & 3) == 0 && i0 + kPerThread <= chi) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(base + i0));
      const float4 b = __ldg(reinterpret_cast<const float4*>(base + i0) + 1);
      lv[0] = a.x; lv[1] = a.y; lv[2] = a.z; lv[3] = a.w;
      lv[4] = b.x; lv[5] = b.y; lv[6] = b.z; lv[7] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < kPerThread; ++k) lv[k] = (i0 + k < chi) ? __ldg(base + i0 + k) : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      fsum += (i0 + k < chi) ? expf((lv[k] - gmax) * invT) : 0.0f;
      pre[k] = fsum;
    }
  }
  const double tsum = (double)fsum;
  // exclusive scan of thread totals across the CTA
  double incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  double wbase = 0.0;
  for (int w = 0; w < warp; ++w) wbase += s_scan[w];
  const double excl = wbase + incl - tsum;
  const double target = s_target;
  int cand = 0x7fffffff;
#pragma unroll
  for (int k = kPerThread - 1; k >= 0; --k) {
    const int i = clo + threadIdx.x * kPerThread + k;
    if (i < chi && excl + (double)pre[k] > target) cand = i;
  }
  if (cand != 0x7fffffff) atomicMin(&s_tok, cand);
  __syncthreads();
  if (threadIdx.x == 0) {
    // Rounding can leave the target just past the chunk's last partial sum:
    // the sample then is the chunk's last logit.
    token[row] = (s_tok != 0x7fffffff) ? s_tok : (chi - 1);
    counters[row] = 0u;
  }
}

// ---- one thread-block cluster per row (the sampler without top-p) ----------------------
// Rows of up to kMaxClusterCtas x 1024 x PER logits: CTA r of a row's cluster
// holds logits [r L, (r+1) L) of it, L = 1024 PER, in registers -- thread t the
// PER consecutive logits from r L + PER t.  The row maximum and the per-CTA
// sums are exchanged through distributed shared memory (two cluster
// barriers), so no partial goes through global memory and no CTA waits on a
// counter.  Every CTA then forms Z, A, H and, from the row state it read at
// entry, the same T (the same operations in the same order); rank 0 writes the
// new state.  The CTA whose range holds u * Z_T scans its own registers for
// the token.
//
// FP64 is a narrow, long-latency pipe on this GPU, so it is kept off every
// per-thread path: sums are FP32 within a thread and a warp, FP64 across warps
// (a shuffle tree) and CTAs; the threshold rule compares means by
// cross-multiplying (sum_a * n_b <= sum_b * n_a) instead of dividing; and the
// token is located in FP64 only down to a warp, then in FP32 within it.
constexpr int kCThreads = 1024;
constexpr int kCWarps = kCThreads / 32;
constexpr int kMaxClusterCtas = 8;                  // portable: every GPC can host such a cluster

__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_dsmem_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

// ---- top-p inside the row's cluster ------------------------------------------------
// Masses are integers, floor(2^a x mscale) with a = (l - max) log2(e) / T, so
// every bin, sum and scan below sees the same numbers and every sum is exact in
// any order: the token depends neither on the cluster's size nor on
// scheduling.  The boundary key is the smallest order key whose inclusive mass
// reaches ceil(top_p Z); a token is kept iff its key is at most the boundary --
// the smallest set of most probable tokens that reaches top_p, every logit tied
// to its least probable member included.  Each thread keeps 2^a mscale of its
// logits in shared memory (dynamic, PER x 4 KB), so the mass is evaluated once.

constexpr int kCand = 4096;            // crossing-bin keys gathered on rank 0, kCand / CS (rounded down to 32) a CTA
constexpr int kSuper = kHistBins / 32; // super-bins of 32 bins: the crossing is found in two 32-wide steps
constexpr int kSubBins = 256;          // rank 0 splits the crossing bin into 256 log-mass sub-bins
constexpr float kBinsPerOctave = 64.0f;

// floor(x) for 0 <= x < 2^63 with integer operations only (a 64-bit conversion
// instruction runs on this GPU's narrow FP64 pipe).  x below 1, from 2^63 up,
// infinite, NaN or negative gives 0.
__device__ __forceinline__ unsigned long long mass_bits(float x) {
  const uint32_t b = __float_as_uint(x);
  const int sh = (int)(b >> 23) - 150;                // x = mant 2^sh for 1 <= x, -23 <= sh <= 39
  const unsigned long long mant = (b & 0x7FFFFFu) | 0x800000u;
  return (b < 0x3F800000u || b >= 0x5F000000u) ? 0ull : (sh >= 0 ? mant << sh : mant >> -sh);
}

// ceil(p z) (up) or floor(p z), exactly, for a float 0 <= p <= 1 and z < 2^63:
// p = mant 2^-sh, the 128-bit product z mant shifted right by sh >= 23.
__device__ __forceinline__ unsigned long long scale_u64(float p, unsigned long long z, bool up) {
  const uint32_t b = __float_as_uint(p);
  const int e = (int)((b >> 23) & 0xFFu);
  const unsigned long long mant = e ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
  const int sh = 150 - (e ? e : 1);
  const unsigned long long lo = z * mant, hi = __umul64hi(z, mant);
  unsigned long long q;
  bool dropped;
  if (sh >= 128) {
    q = 0ull;
    dropped = (hi | lo) != 0ull;
  } else if (sh >= 64) {
    const int s2 = sh - 64;
    q = hi >> s2;
    dropped = lo != 0ull || (s2 > 0 && (hi & ((1ull << s2) - 1ull)) != 0ull);
  } else {
    q = (lo >> sh) | (hi << (64 - sh));
    dropped = (lo & ((1ull << sh) - 1ull)) != 0ull;
  }
  return q + ((up && dropped) ? 1ull : 0ull);
}

// Log-mass bin floor(-64 a): 1/64 octave of mass a bin, the last bin taking
// everything from 32 octaves below the maximum down.  It never decreases as
// the logit falls, so a bin is a contiguous range of order keys.
__device__ __forceinline__ int logmass_bin(float a) {
  const float x = a * -kBinsPerOctave;
  return x < (float)(kHistBins - 1) ? (int)x : kHistBins - 1;
}

// Adds m to bin d of a histogram kept as 32-bit words (low words at d, high
// words at nb + d): shared-memory 32-bit atomics, where a contended 64-bit one
// is many times slower.  A per-CTA bin total stays below 2^62, so the high
// word (the high halves plus the carries) cannot wrap.
__device__ __forceinline__ void hist_add_u64(uint32_t* h32, int nb, int d, unsigned long long m) {
  const uint32_t ml = (uint32_t)m;
  uint32_t mh = (uint32_t)(m >> 32);
  if (ml) {
    const uint32_t old = atomicAdd(&h32[d], ml);
    mh += (old + ml < old) ? 1u : 0u;                 // the low word wrapped
  }
  if (mh) atomicAdd(&h32[nb + d], mh);
}

// Inclusive scan over a warp.
__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  return x;
}
__device__ __forceinline__ unsigned int warp_incl_u32(unsigned int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  return x;
}

// Warp 0: the digit of a 256-bin histogram (32-bit words, low at d, high at
// 256 + d) where the running mass, started at acc, first reaches need.
// Returns the digit in every lane and sets *before to the mass ahead of it.
__device__ __forceinline__ int warp_cross256(const uint32_t* r32, unsigned long long acc, unsigned long long need,
                                             unsigned long long* before) {
  const int lane = threadIdx.x & 31;
  unsigned long long bm[8], lt = 0ull;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    bm[i] = r32[8 * lane + i] | ((unsigned long long)r32[256 + 8 * lane + i] << 32);
    lt += bm[i];
  }
  const unsigned long long li = warp_incl_u64(lt);
  const unsigned hit = __ballot_sync(0xffffffffu, acc + li >= need);
  const int ls = hit ? __ffs(hit) - 1 : 31;
  unsigned long long run = acc + li - lt;
  int dg = 8 * lane + 7;
  bool found = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!found && run + bm[i] >= need) {
      dg = 8 * lane + i;
      found = true;
    }
    if (!found && i < 7) run += bm[i];
  }
  *before = __shfl_sync(0xffffffffu, run, ls);
  return __shfl_sync(0xffffffffu, dg, ls);
}

// The integer mass of logit l at T (cT = log2(e) / T): mass_bits(2^a mscale)
// with a = (l - max) cT.  Every use evaluates the same expression, so every
// bin, sum and scan sees the same integers.
__device__ __forceinline__ unsigned long long cluster_mass(float l, float gm, float cT, float ms) {
  return mass_bits(exp2f((l - gm) * cT) * ms);
}

// The token in this CTA given the boundary key, the target within the CTA's
// kept mass and each thread's kept mass `mine`: token = min{ i : P_i > tloc },
// P the running kept mass in index order (P > u Zk <=> P > floor(u Zk) for
// integers).  The warp from the per-warp kept masses, the lane from the
// threads' totals, then the lane's logits one per lane of the warp.  Returns
// the token in every lane of the chosen warp, -1 elsewhere.  s_v holds logit k
// of thread t at k 1024 + t.
template <int PER>
__device__ __forceinline__ int nucleus_select(const float* s_v, int i0, int hi, float gm, float cT, float ms,
                                              uint32_t kstar, unsigned long long tloc, unsigned long long mine) {
  __shared__ unsigned long long s_pw[kCWarps];
  __shared__ int s_wsel;
  __shared__ unsigned long long s_wtl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long ws = warp_sum_u64(mine);
  if (lane == 0) s_pw[warp] = ws;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long wt = s_pw[lane];
    const unsigned long long wi = warp_incl_u64(wt);
    const unsigned hit = __ballot_sync(0xffffffffu, wi > tloc);
    const int wsel = hit ? __ffs(hit) - 1 : 31;
    const unsigned long long wb = __shfl_sync(0xffffffffu, wi - wt, wsel);
    if (lane == 0) {
      s_wsel = wsel;
      s_wtl = tloc - wb;
    }
  }
  __syncthreads();
  if (warp != s_wsel) return -1;
  const unsigned long long tl = s_wtl;
  const unsigned long long incl = warp_incl_u64(mine);
  const unsigned hit = __ballot_sync(0xffffffffu, incl > tl);
  const int lsel = hit ? __ffs(hit) - 1 : 31;
  // lane j takes logit j of lane lsel
  const unsigned long long base = __shfl_sync(0xffffffffu, incl - mine, lsel);
  const int is = __shfl_sync(0xffffffffu, i0, lsel);
  const bool live = lane < PER && is + lane < hi;
  const float lj = live ? s_v[lane * kCThreads + 32 * warp + lsel] : 0.0f;
  const unsigned long long mj = (live && nucleus_key(lj) <= kstar) ? cluster_mass(lj, gm, cT, ms) : 0ull;
  const unsigned long long run = base + warp_incl_u64(mj);
  const unsigned h2 = __ballot_sync(0xffffffffu, live && run > tl);
  const unsigned lv = __ballot_sync(0xffffffffu, live);
  // exact sums always find it; else the lane's last logit
  return min(is + (h2 ? __ffs(h2) - 1 : (lv ? 31 - __clz(lv) : 0)), hi - 1);
}

// The same, each thread's kept mass summed over all its logits.
template <int PER>
__device__ __forceinline__ int nucleus_pick(const float* s_v, int i0, int hi, float gm, float cT, float ms,
                                            uint32_t kstar, unsigned long long tloc) {
  unsigned long long mine = 0ull;
#pragma unroll 4
  for (int k = 0; k < PER; ++k) {
    const float l = s_v[k * kCThreads + threadIdx.x];
    if (i0 + k < hi && nucleus_key(l) <= kstar) mine += cluster_mass(l, gm, cT, ms);
  }
  return nucleus_select<PER>(s_v, i0, hi, gm, cT, ms, kstar, tloc, mine);
}

// The boundary key by a three-level radix search over the order keys (11, 11
// and 10 bits) across the cluster.  Per level: each CTA bins its own logits'
// masses; after a cluster barrier each CTA sums a 1/CS slice of the bins over
// every CTA and pushes its slice total; after a second barrier the CTA whose
// slice holds the crossing finds the digit and pushes it to every CTA; a third
// barrier publishes it.  Then the CTAs' kept masses are exchanged and the CTA
// holding floor(u Zk) picks the token.  Used when the crossing log-mass bin
// holds more keys than the gather below has room for (large ties); kept out
// of line, off the common path's code.
template <int PER>
__device__ __noinline__ int cluster_nucleus_radix(const float* s_v, int i0, int hi, float gm, float cT, float ms,
                                                  float top_p, uint32_t rank, int CS, float u_row,
                                                  unsigned long long* s_hist) {
  __shared__ unsigned long long s_slice[kMaxClusterCtas];  // per CTA: its slice total (levels), its kept mass
  __shared__ unsigned long long s_res[3];          // the level's digit, mass below it, mass of its bin
  __shared__ unsigned long long s_w64[kCWarps], s_wex[kCWarps];
  __shared__ int s_pick;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  uint32_t* h32 = reinterpret_cast<uint32_t*>(s_hist);
  unsigned int prefix = 0;
  unsigned long long below = 0ull, target = 0ull, binmass = 0ull;
#pragma unroll 1
  for (int level = 0; level < 3; ++level) {
    const int nb = level == 2 ? 1024 : kHistBins;
    for (int b = t; b < kHistBins; b += kCThreads) s_hist[b] = 0ull;
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < PER; ++k) {
      const float l = s_v[k * kCThreads + t];
      if (i0 + k < hi) {
        const uint32_t key = nucleus_key(l);
        const bool match = level == 0 ? true : level == 1 ? (key >> 21) == prefix : (key >> 10) == prefix;
        if (match) {
          const uint32_t d = level == 0 ? key >> 21 : level == 1 ? (key >> 10) & 0x7FFu : key & 0x3FFu;
          hist_add_u64(h32, kHistBins, (int)d, cluster_mass(l, gm, cT, ms));
        }
      }
    }
    __syncthreads();
    {                                               // fold the words into 64-bit bins in place
      const unsigned long long c0 = h32[t] | ((unsigned long long)h32[kHistBins + t] << 32);
      const unsigned long long c1 =
          h32[t + kCThreads] | ((unsigned long long)h32[kHistBins + t + kCThreads] << 32);
      __syncthreads();
      s_hist[t] = c0;
      s_hist[t + kCThreads] = c1;
    }
    cluster_sync();                                 // every CTA's histogram is complete
    // This CTA's slice of the row histogram, bins [rank sl, rank sl + sl):
    // thread t holds the `per` consecutive bins from rank sl + t per (per is 1,
    // or 2 when one CTA covers 2048 bins).
    const int sl = (nb + CS - 1) / CS;
    const int per = (sl + kCThreads - 1) / kCThreads;
    const int send = min(nb, ((int)rank + 1) * sl);  // end of this CTA's slice
    const int b0 = (int)rank * sl + t * per;
    unsigned long long bins[2] = {0ull, 0ull};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int bb = b0 + j;
      if (j < per && bb < send) {
        unsigned long long x[kMaxClusterCtas];
#pragma unroll
        for (int r = 0; r < kMaxClusterCtas; ++r) x[r] = r < CS ? ld_dsmem_u64(dsmem_addr(&s_hist[bb], (uint32_t)r)) : 0ull;
#pragma unroll
        for (int r = 0; r < kMaxClusterCtas; ++r) bins[j] += x[r];
      }
    }
    const unsigned long long bin = bins[0] + bins[1];   // this thread's total
    const unsigned long long ws = warp_sum_u64(bin);
    if (lane == 0) s_w64[warp] = ws;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long tot = warp_sum_u64(s_w64[lane]);
      if (lane < CS) st_dsmem_u64(dsmem_addr(&s_slice[rank], (uint32_t)lane), tot);
      __syncwarp();
    }
    cluster_sync();                                 // slice totals published; peers are done with s_hist
    if (level == 0) {
      unsigned long long z = 0ull;
      for (int r = 0; r < CS; ++r) z += s_slice[r];
      // z >= 1: the maximum's mass is mscale; the target is in [1, z]
      const unsigned long long tg = scale_u64(top_p, z, true);
      target = tg < 1ull ? 1ull : (tg > z ? z : tg);
    }
    // the slice holding the crossing: the first whose running total reaches the target
    int rstar = CS - 1;
    unsigned long long pre = below;
    for (int r = 0; r < CS; ++r) {
      if (pre + s_slice[r] >= target) {
        rstar = r;
        break;
      }
      pre += s_slice[r];
    }
    if ((int)rank == rstar) {
      // exclusive scan of the threads' totals in bin order
      const unsigned long long incl = warp_incl_u64(bin);
      if (lane == 31) s_w64[warp] = incl;
      if (t == 0) s_pick = 0x7fffffff;
      __syncthreads();
      if (warp == 0) {
        const unsigned long long wv = s_w64[lane];
        s_wex[lane] = warp_incl_u64(wv) - wv;
      }
      __syncthreads();
      const unsigned long long excl = pre + s_wex[warp] + incl - bin;
      // the thread whose bins hold the crossing
      if (b0 < send && excl + bin >= target && excl < target) atomicMin(&s_pick, t);
      __syncthreads();
      // The levels see the same integers, so the range chosen at the level
      // before reaches the target; the fallback (the slice's last bin) is not
      // reached.
      const int last_t = (send - 1 - (int)rank * sl) / per;
      const int tp = s_pick != 0x7fffffff ? s_pick : last_t;
      if (t == tp) {
        // within the thread's bins: the first that reaches the target, else
        // its last bin
        const bool two = per == 2 && b0 + 1 < send;
        const bool first = !two || excl + bins[0] >= target;
        const int bsel = first ? b0 : b0 + 1;
        const unsigned long long bm = first ? bins[0] : bins[1];
        const unsigned long long ex = first ? excl : excl + bins[0];
        for (int r = 0; r < CS; ++r) {
          st_dsmem_u64(dsmem_addr(&s_res[0], (uint32_t)r), (unsigned long long)bsel);
          st_dsmem_u64(dsmem_addr(&s_res[1], (uint32_t)r), ex);
          st_dsmem_u64(dsmem_addr(&s_res[2], (uint32_t)r), bm);
        }
      }
      __syncwarp();
    }
    cluster_sync();                                 // the digit is everywhere
    const unsigned int digit = (unsigned int)s_res[0];
    below = s_res[1];
    binmass = s_res[2];
    prefix = level == 0 ? digit : level == 1 ? (prefix << 11) | digit : (prefix << 10) | digit;
  }
  const unsigned int kstar = prefix;               // the boundary key
  const unsigned long long zk = below + binmass;   // the nucleus's mass

  // ---- the CTAs' kept masses, then the CTA holding floor(u Zk) ----
  unsigned long long mine = 0ull;
#pragma unroll 1
  for (int k = 0; k < PER; ++k) {
    const float l = s_v[k * kCThreads + t];
    if (i0 + k < hi && nucleus_key(l) <= kstar) mine += cluster_mass(l, gm, cT, ms);
  }
  const unsigned long long ws = warp_sum_u64(mine);
  if (lane == 0) s_w64[warp] = ws;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long tot = warp_sum_u64(s_w64[lane]);
    if (lane < CS) st_dsmem_u64(dsmem_addr(&s_slice[rank], (uint32_t)lane), tot);
    __syncwarp();
  }
  cluster_sync();
  unsigned long long tgt = scale_u64(u_row, zk, false);   // floor(u Zk) in [0, Zk)
  if (tgt >= zk) tgt = zk - 1ull;
  int rstar = CS - 1;
  unsigned long long pre = 0ull;
  for (int r = 0; r < CS; ++r) {
    if (pre + s_slice[r] > tgt) {
      rstar = r;
      break;
    }
    pre += s_slice[r];
  }
  if ((int)rank != rstar) return -1;
  return nucleus_select<PER>(s_v, i0, hi, gm, cT, ms, kstar, tgt - pre, mine);
}

// Rank 0, when more than 32 gathered keys share the crossing sub-bin (ties,
// or a dense bin): the boundary key by eight key bits a round over the
// sub-bin's keys, from acc (the mass of the gathered keys in lower sub-bins).
// Every thread of rank 0 calls it; out of line, off the common path's code.
__device__ __noinline__ uint32_t gathered_radix(const uint32_t* s_ck, const unsigned long long* s_cm,
                                                const uint8_t* s_cb, const unsigned int* s_ccnt, int Cr, int CS,
                                                int sbs, unsigned long long acc, unsigned long long need,
                                                unsigned long long* s_rh, unsigned long long* s_sel) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  uint32_t* r32 = reinterpret_cast<uint32_t*>(s_rh);
  uint32_t prefix = 0u;
#pragma unroll 1
  for (int round = 0; round < 4; ++round) {
    const int sh = 24 - 8 * round;
    if (t < kSubBins) s_rh[t] = 0ull;
    __syncthreads();
    for (int r = 0; r < CS; ++r) {
      const int n = (int)s_ccnt[r];
      for (int j = t; j < n; j += kCThreads) {
        const int s = r * Cr + j;
        const uint32_t key = s_ck[s];
        if ((int)s_cb[s] == sbs && s_cm[s] && (round == 0 || (key >> (sh + 8)) == prefix))
          hist_add_u64(r32, kSubBins, (int)((key >> sh) & 0xFFu), s_cm[s]);
      }
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long before;
      const int dg = warp_cross256(r32, acc, need, &before);
      if (lane == 0) {
        s_sel[0] = (unsigned long long)dg;
        s_sel[1] = before;
      }
    }
    __syncthreads();
    prefix = (prefix << 8) | (uint32_t)s_sel[0];
    acc = s_sel[1];
    __syncthreads();
  }
  return prefix;
}

// Top-p inside the row's cluster (every CTA of the cluster calls it, with T
// known), in three cluster barriers:
//  1. each CTA bins its logits' masses by log-mass (1/64 octave a bin, exact
//     integer totals) in shared memory, with the totals of 64 super-bins of
//     32 bins, pushed to every CTA; barrier;
//  2. in every CTA one warp finds the super-bin where the running mass
//     reaches ceil(top_p Z), then reads its 32 bins of every CTA and finds the
//     crossing bin -- the same in every CTA; each CTA sends rank 0 its mass
//     before that bin and, for each of its logits inside it, the order key,
//     the mass and a sub-bin (1/256 of the bin); barrier;
//  3. rank 0 finds the boundary key among the gathered ones: a histogram of
//     the 256 sub-bins, then an exact comparison of the keys in the crossing
//     sub-bin (a radix search over the key bits when that holds more than 32);
//     it forms each CTA's kept mass, locates floor(u Zk) and tells the CTA
//     that holds it; barrier; that CTA picks the token.  While rank 0
//     searches, the other CTAs sum each thread's mass before the crossing bin,
//     so the pick only adds the thread's logits inside it.
// A bin spans 1/64 octave of probability, so the crossing bin holds few
// logits; if some CTA finds more than its share of kCand, every CTA runs the
// radix search above instead.
//
// The logits are read from shared memory (s_v: logit k of thread t at
// k 1024 + t), not registers, which the 1024-thread CTA has 64 of a thread.
// Dynamic shared memory: the logits, then rank 0's gathered masses, keys and
// sub-bins.
template <int PER>
constexpr size_t cluster_nucleus_smem() {
  return (size_t)PER * kCThreads * sizeof(float) + (size_t)kCand * (sizeof(unsigned long long) + sizeof(uint32_t) + 1);
}

template <int PER>
__device__ __forceinline__ int cluster_nucleus(const float* s_v, int i0, int hi, float gm, float cT, const Params& p,
                                               uint32_t rank, int CS, float u_row) {
  static_assert(kHistBins == 2 * kCThreads && kSuper == 64, "two bins a thread, two super-bins a lane");
  static_assert(PER <= 32, "one match bit (and one lane of the pick) a logit");
  static_assert(kCThreads >= kSubBins && kCand % kCThreads == 0, "one sub-bin a thread");
  __shared__ __align__(16) unsigned long long s_hist[kHistBins];  // this CTA's bins (32-bit words while binning)
  __shared__ unsigned long long s_sup[kMaxClusterCtas][kSuper];   // every CTA's super-bin totals
  __shared__ unsigned int s_ccnt[kMaxClusterCtas];      // rank 0: how many logits CTA r sent
  __shared__ unsigned long long s_cmass[kMaxClusterCtas];  // rank 0: CTA r's mass before the crossing bin
  __shared__ unsigned long long s_kept[kMaxClusterCtas];   // rank 0: CTA r's kept mass
  __shared__ unsigned long long s_w64[kCWarps];
  __shared__ unsigned int s_wcnt[kCWarps];
  __shared__ unsigned long long s_x[3];                 // the crossing bin, the mass before it, the target
  __shared__ unsigned long long s_rh[kSubBins];         // rank 0: sub-bin / digit masses (32-bit words)
  __shared__ unsigned int s_rc[kSubBins];               // rank 0: sub-bin counts
  __shared__ uint32_t s_k32[32];                        // rank 0: the crossing sub-bin's keys ...
  __shared__ unsigned long long s_m32[32];              // ... and masses
  __shared__ unsigned int s_n32;
  __shared__ unsigned long long s_sel[3];               // rank 0: sub-bin, mass before it, boundary key
  __shared__ unsigned long long s_fin[2];               // from rank 0: the boundary key, the target in this CTA
  __shared__ unsigned int s_status;                     // from rank 0: 0 done, 1 pick the token, 2 radix search
  extern __shared__ __align__(16) unsigned char s_dyn[];
  unsigned long long* s_cm = reinterpret_cast<unsigned long long*>(s_dyn + (size_t)PER * kCThreads * sizeof(float));
  uint32_t* s_ck = reinterpret_cast<uint32_t*>(s_cm + kCand);
  uint8_t* s_cb = reinterpret_cast<uint8_t*>(s_ck + kCand);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const float ms = p.mscale;
  uint32_t* h32 = reinterpret_cast<uint32_t*>(s_hist);
  const int b0 = 2 * t;                                 // this thread's two bins

  // ---- 1. this CTA's log-mass histogram and super-bin totals ----
  s_hist[b0] = 0ull;
  s_hist[b0 + 1] = 0ull;
  __syncthreads();
#pragma unroll 4
  for (int k = 0; k < PER; ++k) {
    const float a = (s_v[k * kCThreads + t] - gm) * cT;
    const unsigned long long m = mass_bits(exp2f(a) * ms);
    if (i0 + k < hi && m) hist_add_u64(h32, kHistBins, logmass_bin(a), m);
  }
  __syncthreads();
  {                                                     // fold the words into 64-bit bins in place
    const unsigned long long c0 = h32[b0] | ((unsigned long long)h32[kHistBins + b0] << 32);
    const unsigned long long c1 = h32[b0 + 1] | ((unsigned long long)h32[kHistBins + b0 + 1] << 32);
    __syncthreads();
    s_hist[b0] = c0;
    s_hist[b0 + 1] = c1;
    // lanes 0-15 of warp w hold super-bin 2w, lanes 16-31 super-bin 2w + 1:
    // pushed to every CTA of the cluster
    unsigned long long sp = c0 + c1;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sp += __shfl_xor_sync(0xffffffffu, sp, o);
    if ((lane & 15) == 0)
      for (int r = 0; r < CS; ++r) st_dsmem_u64(dsmem_addr(&s_sup[rank][2 * warp + (lane >> 4)], (uint32_t)r), sp);
  }
  cluster_sync();                                       // every CTA's bins and super-bin totals are in place

  // ---- 2. warp 0: the crossing super-bin, then the crossing bin ----
  if (warp == 0) {
    unsigned long long sa = 0ull, sb = 0ull;
#pragma unroll
    for (int r = 0; r < kMaxClusterCtas; ++r) {
      if (r < CS) {
        sa += s_sup[r][2 * lane];
        sb += s_sup[r][2 * lane + 1];
      }
    }
    const unsigned long long lt = sa + sb;
    const unsigned long long li = warp_incl_u64(lt);
    const unsigned long long z = __shfl_sync(0xffffffffu, li, 31);   // >= 1: the maximum's mass is mscale
    unsigned long long target = scale_u64(p.top_p, z, true);
    target = target < 1ull ? 1ull : (target > z ? z : target);
    const unsigned h1 = __ballot_sync(0xffffffffu, li >= target);
    const int l1 = h1 ? __ffs(h1) - 1 : 31;
    const unsigned long long ex1 = __shfl_sync(0xffffffffu, li - lt, l1);
    const unsigned long long sa1 = __shfl_sync(0xffffffffu, sa, l1);
    const bool first = ex1 + sa1 >= target;
    const int S = 2 * l1 + (first ? 0 : 1);
    const unsigned long long bS = first ? ex1 : ex1 + sa1;   // mass before super-bin S
    unsigned long long fb = 0ull;
    {
      unsigned long long q[kMaxClusterCtas];
#pragma unroll
      for (int r = 0; r < kMaxClusterCtas; ++r) q[r] = r < CS ? ld_dsmem_u64(dsmem_addr(&s_hist[32 * S + lane], (uint32_t)r)) : 0ull;
#pragma unroll
      for (int r = 0; r < kMaxClusterCtas; ++r) fb += q[r];
    }
    const unsigned long long fi = warp_incl_u64(fb);
    const unsigned h2 = __ballot_sync(0xffffffffu, bS + fi >= target);
    const int l2 = h2 ? __ffs(h2) - 1 : 31;
    if (lane == l2) {
      s_x[0] = (unsigned long long)(32 * S + l2);
      s_x[1] = bS + fi - fb;
      s_x[2] = target;
    }
  }
  __syncthreads();
  const int dstar = (int)s_x[0];
  const unsigned long long below = s_x[1], target = s_x[2];

  // ---- this CTA's mass before the crossing bin and its logits inside it -> rank 0 ----
  // -64 a is an exact scaling, so the bin test d <= -64 a < d + 1 is
  // a <= -d/64 and a > -(d + 1)/64 (the last bin has no lower end); NaN is
  // in neither, and has no mass.
  const int Cr = (kCand / CS) & ~31;                    // logits a CTA may send
  const unsigned long long mb = (b0 < dstar ? s_hist[b0] : 0ull) + (b0 + 1 < dstar ? s_hist[b0 + 1] : 0ull);
  const float a_hi = (float)dstar * (-1.0f / kBinsPerOctave);
  const float a_lo = dstar == kHistBins - 1 ? -INFINITY : (float)(dstar + 1) * (-1.0f / kBinsPerOctave);
  uint32_t match = 0u, lower = 0u;                      // logits in / before the crossing bin
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const float a = (s_v[k * kCThreads + t] - gm) * cT;
    if (i0 + k < hi) {
      if (a <= a_hi && a > a_lo) match |= 1u << k;
      if (a > a_hi) lower |= 1u << k;
    }
  }
  const unsigned int cnt = __popc(match);
  const unsigned int ci = warp_incl_u32(cnt);
  const unsigned long long mw = warp_sum_u64(mb);
  if (lane == 31) s_wcnt[warp] = ci;
  if (lane == 0) s_w64[warp] = mw;
  __syncthreads();
  if (warp == 0) {
    const unsigned int wc = s_wcnt[lane];
    const unsigned int wci = warp_incl_u32(wc);
    const unsigned long long mt = warp_sum_u64(s_w64[lane]);
    __syncwarp();
    s_wcnt[lane] = wci - wc;
    if (lane == 31) {
      st_dsmem_u32(dsmem_addr(&s_ccnt[rank], 0u), wci);
      st_dsmem_u64(dsmem_addr(&s_cmass[rank], 0u), mt);
    }
  }
  __syncthreads();
  if (match) {
    unsigned int slot = s_wcnt[warp] + ci - cnt;
    uint32_t mm = match;
    while (mm) {
      const int k = __ffs(mm) - 1;
      mm &= mm - 1u;
      if (slot < (unsigned)Cr) {
        const int j = (int)rank * Cr + (int)slot;
        const float l = s_v[k * kCThreads + t];
        const float a = (l - gm) * cT;
        // sub-bin: the fraction of -64 a past the bin's start, x 256 (exact steps)
        const float f = (a * -kBinsPerOctave - (float)dstar) * (float)kSubBins;
        const uint32_t sbin = f < (float)(kSubBins - 1) ? (uint32_t)f : (uint32_t)(kSubBins - 1);
        st_dsmem_u64(dsmem_addr(&s_cm[j], 0u), mass_bits(exp2f(a) * ms));
        st_dsmem_u32(dsmem_addr(&s_ck[j], 0u), nucleus_key(l));
        st_dsmem_u8(dsmem_addr(&s_cb[j], 0u), sbin);
      }
      ++slot;
    }
  }
  cluster_sync();                                       // the gathered logits and masses are on rank 0

  // ---- 3. rank 0: the boundary key, the kept masses, the CTA holding the sample ----
  unsigned long long mine = 0ull;                       // this thread's mass before the crossing bin
  if (rank == 0) {
    bool over = false;
    for (int r = 0; r < CS; ++r) over |= s_ccnt[r] > (unsigned)Cr;
    if (over) {
      if (t < CS) st_dsmem_u32(dsmem_addr(&s_status, (uint32_t)t), 2u);
    } else {
      constexpr int kQ = kCand / kCThreads;
      uint32_t ck[kQ];
      unsigned long long cm[kQ];
      int csb[kQ];
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int s = t + q * kCThreads;
        int r = 0;
#pragma unroll
        for (int i = 1; i < kMaxClusterCtas; ++i) r += s >= i * Cr ? 1 : 0;
        const uint32_t kk = s_ck[s];                    // (slots past a CTA's count hold stale words)
        const unsigned long long mm = s_cm[s];
        const int bb = (int)s_cb[s];
        const bool ok = r < CS && s - r * Cr < (int)s_ccnt[r];
        ck[q] = ok ? kk : 0xFFFFFFFFu;
        cm[q] = ok ? mm : 0ull;
        csb[q] = ok ? bb : -1;
      }
      // The smallest key K with (mass of gathered keys <= K) >= target - below.
      // Sub-bins never decrease with the key, so every key of a lower sub-bin
      // is below every key of a higher one.
      const unsigned long long need = target - below;  // >= 1: the bins before the crossing fall short
      uint32_t* r32 = reinterpret_cast<uint32_t*>(s_rh);
      if (t < kSubBins) {
        s_rh[t] = 0ull;
        s_rc[t] = 0u;
      }
      if (t == 0) s_n32 = 0u;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        if (csb[q] >= 0) {
          if (cm[q]) hist_add_u64(r32, kSubBins, csb[q], cm[q]);
          atomicAdd(&s_rc[csb[q]], 1u);
        }
      }
      __syncthreads();
      if (warp == 0) {
        unsigned long long acc;
        const int sbs = warp_cross256(r32, 0ull, need, &acc);
        if (lane == 0) {
          s_sel[0] = (unsigned long long)sbs;
          s_sel[1] = acc;
        }
      }
      __syncthreads();
      const int sbs = (int)s_sel[0];
      const unsigned long long acc = s_sel[1];
      const unsigned int n32 = s_rc[sbs];
      uint32_t kstar;
      if (n32 <= 32u) {
        // the crossing sub-bin's keys, compared exactly in one warp
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          if (csb[q] == sbs) {
            const unsigned int j = atomicAdd(&s_n32, 1u);
            s_k32[j] = ck[q];
            s_m32[j] = cm[q];
          }
        }
        __syncthreads();
        if (warp == 0) {
          const bool has = (unsigned)lane < n32;
          const uint32_t kl = has ? s_k32[lane] : 0xFFFFFFFFu;
          const unsigned long long ml = has ? s_m32[lane] : 0ull;
          unsigned long long cum = 0ull;                // mass of the sub-bin's keys <= kl
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t kj = __shfl_sync(0xffffffffu, kl, j);
            const unsigned long long mj = __shfl_sync(0xffffffffu, ml, j);
            if (kj <= kl) cum += mj;
          }
          uint32_t best = (has && acc + cum >= need) ? kl : 0xFFFFFFFFu;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
          if (lane == 0) s_sel[2] = best;
        }
        __syncthreads();
        kstar = (uint32_t)s_sel[2];
      } else {
        kstar = gathered_radix(s_ck, s_cm, s_cb, s_ccnt, Cr, CS, sbs, acc, need, s_rh, s_sel);
      }
      // each CTA's kept mass: its mass before the bin + its gathered keys <= kstar
      // (warp r sums CTA r's range)
      if (warp < CS) {
        const int n = (int)s_ccnt[warp];
        unsigned long long kw = 0ull;
        for (int j = lane; j < n; j += 32)
          if (s_ck[warp * Cr + j] <= kstar) kw += s_cm[warp * Cr + j];
        kw = warp_sum_u64(kw);
        if (lane == 0) s_kept[warp] = s_cmass[warp] + kw;
      }
      __syncthreads();
      if (warp == 0) {
        // zk >= target >= 1; the sample is floor(u zk) in [0, zk), in the first
        // CTA whose running kept mass passes it
        const unsigned long long kr = lane < CS ? s_kept[lane] : 0ull;
        const unsigned long long ki = warp_incl_u64(kr);
        const unsigned long long zk = __shfl_sync(0xffffffffu, ki, 31);
        unsigned long long tgt = scale_u64(u_row, zk, false);
        if (tgt >= zk) tgt = zk - 1ull;
        const unsigned hr = __ballot_sync(0xffffffffu, lane < CS && ki > tgt);
        const int rstar = hr ? __ffs(hr) - 1 : CS - 1;
        if (lane == rstar) {
          st_dsmem_u64(dsmem_addr(&s_fin[0], (uint32_t)rstar), (unsigned long long)kstar);
          st_dsmem_u64(dsmem_addr(&s_fin[1], (uint32_t)rstar), tgt - (ki - kr));
        }
        if (lane < CS) st_dsmem_u32(dsmem_addr(&s_status, (uint32_t)lane), lane == rstar ? 1u : 0u);
      }
    }
  } else {
    uint32_t lw = lower;
    while (lw) {
      const int k = __ffs(lw) - 1;
      lw &= lw - 1u;
      mine += cluster_mass(s_v[k * kCThreads + t], gm, cT, ms);
    }
  }
  cluster_sync();                                       // the verdict is in every CTA
  const unsigned int status = s_status;
  if (status == 2u) return cluster_nucleus_radix<PER>(s_v, i0, hi, gm, cT, ms, p.top_p, rank, CS, u_row, s_hist);
  if (status != 1u) return -1;
  const uint32_t kstar = (uint32_t)s_fin[0];
  if (rank == 0) {
    uint32_t lw = lower;
    while (lw) {
      const int k = __ffs(lw) - 1;
      lw &= lw - 1u;
      mine += cluster_mass(s_v[k * kCThreads + t], gm, cT, ms);
    }
  }
  uint32_t mw2 = match;
  while (mw2) {
    const int k = __ffs(mw2) - 1;
    mw2 &= mw2 - 1u;
    const float l = s_v[k * kCThreads + t];
    if (nucleus_key(l) <= kstar) mine += cluster_mass(l, gm, cT, ms);
  }
  return nucleus_select<PER>(s_v, i0, hi, gm, cT, ms, kstar, s_fin[1], mine);
}

template <int PER, bool NUC>
__global__ void __launch_bounds__(kCThreads, 1) reset_cluster_kernel(const float* __restrict__ logits, int V, int CS,
                                                                      const uint8_t* __restrict__ step_start,
                                                                      const float* __restrict__ u, uint8_t* state,
                                                                      int stride, Params p, int32_t* token,
                                                                      float* H_out, float* T_out) {
  constexpr int kCover = kCThreads * PER;
  // e^x evaluated as 2^(x log2 e): one multiply and the hardware exp2.  The
  // rounding of x log2 e gives a relative error of about |x| 1.2e-7 per term,
  // so ~1e-7 of Z for the terms near the maximum that make up Z.
  constexpr float kLog2e = 1.4426950408889634f;
  __shared__ float s_wmax[kCWarps];
  __shared__ float s_wred[5][kCWarps];              // per warp: n0, z1, a1, Z_T at T_low, at T_high
  __shared__ float s_peer[kMaxClusterCtas][6];      // per CTA: its maximum, then the same five sums
  __shared__ double s_ring_rest;                    // the window's other w - 1 entropies
  __shared__ RowState s_st;
  __shared__ float s_T, s_gm;
  __shared__ int s_warp, s_rstar, s_zi;
  __shared__ float s_tl;

  const uint32_t rank = cluster_ctarank();
  const int row = blockIdx.x / CS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* base = logits + (size_t)row * V;
  const int lo = (int)rank * kCover;
  const int hi = min(V, lo + kCover);
  const int i0 = lo + threadIdx.x * PER;
  // Peers may write into this CTA's shared memory only once it runs: arrive
  // now, wait just before the first remote store.
  if (CS > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  float v[PER];
  if ((V & 3) == 0 && (PER & 3) == 0 && i0 + PER <= hi) {   // row start 16-byte aligned, all in range
#pragma unroll
    for (int k = 0; k < PER / 4; ++k) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(base + i0) + k);
      v[4 * k] = q.x;
      v[4 * k + 1] = q.y;
      v[4 * k + 2] = q.z;
      v[4 * k + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = (i0 + k < hi) ? __ldg(base + i0 + k) : -INFINITY;
  }
  extern __shared__ __align__(16) unsigned char s_dyn[];
  if constexpr (NUC) {                              // top-p reads the logits from shared memory
    float* s_v = reinterpret_cast<float*>(s_dyn);
#pragma unroll
    for (int k = 0; k < PER; ++k) s_v[k * kCThreads + threadIdx.x] = v[k];
  }

  // ---- this CTA's maximum: the sums below are relative to it, and thread 0
  // rescales each CTA's sums to the row maximum, so the maximum and the sums
  // cross the cluster in one exchange ----
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < PER; ++k) mx = fmaxf(mx, v[k]);
  mx = warp_max(mx);
  if (lane == 0) s_wmax[warp] = mx;
  __syncthreads();
  mx = warp_max(s_wmax[lane]);                      // every warp reduces the 32 warp maxima itself
  const float mb = (mx == -INFINITY) ? 0.0f : mx;   // a CTA of -inf logits sums zeros

  // The row state (every CTA derives T from it; rank 0 updates it after the
  // last cluster barrier, when every CTA has read it): the last warp reads it,
  // its lanes the window ring in parallel (w <= 256: up to 8 entries a lane).
  if (warp == kCWarps - 1) {
    const RowState* st = reinterpret_cast<const RowState*>(state + (size_t)row * stride);
    const RowState r = *st;
    double rest = 0.0;
    if (r.w == p.w && r.t + 1 > p.w) {
      const double* ring = reinterpret_cast<const double*>(st + 1);
      const int slot = r.t % p.w;
      for (int i = lane; i < p.w; i += 32)
        if (i != slot) rest += ring[i];
    }
    rest = warp_sum_d(rest);
    if (lane == 0) {
      s_st = r;
      s_ring_rest = rest;
    }
  }

  // ---- per-thread sums relative to the row maximum (FP32).  Logits equal to
  // the maximum are counted, not summed; at T_high = 1 the T_high sum is the
  // T = 1 sum.  A thread keeps its Z_T for both temperatures for the scan ----
  const float cl = kLog2e * (1.0f / p.t_low), ch = kLog2e * (1.0f / p.t_high);
  const bool th_one = (p.t_high == 1.0f);
  float n0 = 0.f, z1 = 0.f, a1 = 0.f, zl = 0.f, zh = 0.f;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    if (i0 + k < hi) {
      const float s = v[k] - mb;
      if (s == 0.0f) {
        n0 += 1.0f;
      } else {
        const float e = exp2f(s * kLog2e);
        z1 += e;
        if (e > 0.0f) a1 += e * s;                  // a -inf logit adds nothing (not 0 x -inf)
      }
      if constexpr (!NUC) {                         // top-p forms its own masses at the chosen T
        zl += exp2f(s * cl);
        if (!th_one) zh += exp2f(s * ch);
      }
    }
  }
  if (th_one) zh = n0 + z1;
  const float my_zl = zl, my_zh = zh;
  float f[5] = {n0, z1, a1, zl, zh};
#pragma unroll
  for (int i = 0; i < 5; ++i) f[i] = warp_sum(f[i]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 5; ++i) s_wred[i][warp] = f[i];
  }
  __syncthreads();
  if (CS > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer runs: remote stores allowed
  if (warp == 0) {                                  // this CTA's maximum and five sums over its 32 warps
    float g[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) g[i] = warp_sum(s_wred[i][lane]);
    if (lane < 6) {
      const float acc = lane == 0 ? mx : lane == 1 ? g[0] : lane == 2 ? g[1] : lane == 3 ? g[2] : lane == 4 ? g[3] : g[4];
      if (CS > 1) {
        for (int r = 0; r < CS; ++r) st_dsmem_f32(dsmem_addr(&s_peer[rank][lane], r), acc);
      } else {
        s_peer[0][lane] = acc;
      }
    }
    __syncwarp();
  }
  if (CS > 1) cluster_sync();
  else __syncthreads();

  // ---- the row maximum, H, the state rule and T (warp 0; every CTA the
  // same).  Lane r rescales CTA r's FP32 sums by e^(its maximum - the row
  // maximum), its A also gaining that difference x its Z; the lanes' sums are
  // reduced in a fixed order.  Z - 1 is (the row maxima counted - 1) + the
  // rest, so a nearly one-hot row keeps its relative precision.  Lane 0
  // applies the state rule, with FP64 sums ----
  if (warp == 0) {
    const bool has = lane < CS;
    const float mr = has ? s_peer[lane][0] : -INFINITY;
    const float gmax = warp_max(mr);
    const bool live = has && mr != -INFINITY;       // a CTA of only -inf logits has no mass
    const float d = live ? mr - gmax : 0.0f;
    const float fl = live ? exp2f(d * cl) : 0.0f, fh = live ? exp2f(d * ch) : 0.0f;
    float c_cnt = 0.f, c_rest = 0.f, c_A = 0.f;
    if (live) {
      const float n0r = s_peer[lane][1], z1r = s_peer[lane][2], a1r = s_peer[lane][3];
      if (d == 0.0f) {
        c_cnt = n0r;
        c_rest = z1r;
        c_A = a1r;
      } else {
        const float f = exp2f(d * kLog2e), zr = n0r + z1r;
        c_rest = f * zr;
        c_A = f * (a1r + d * zr);
      }
    }
    const float zlr = live ? fl * s_peer[lane][4] : 0.0f, zhr = live ? fh * s_peer[lane][5] : 0.0f;
    const float cnt = warp_sum(c_cnt), rest = warp_sum(c_rest), A = warp_sum(c_A);
    const float ztl = warp_sum(zlr), zth = warp_sum(zhr);
    int low = 0;
    if (lane == 0) {
      const float zm1 = (cnt - 1.0f) + rest;
      const double H = (double)(log1pf(zm1) - A / (1.0f + zm1));
      RowState ns = s_st;
      const int w = p.w;
      const bool state_ok = (ns.w == w);
      int t1 = 0, j = 0;
      if (state_ok) {
        if (ns.t == 0 || (step_start && step_start[row])) {
          ns.j = 0;
          ns.step_sum = 0.0;
        }
        ns.glob_sum += H;
        ns.step_sum += H;
        t1 = ns.t + 1;
        j = ns.j;
        // The window mean is wsum / wn: the whole history while t1 <= w.
        const double wsum = (t1 > w) ? s_ring_rest + H : ns.glob_sum;
        const int wn = (t1 > w) ? w : t1;
        // H_step = ssum / sn; H_bar = glob_sum / t1.  Means are compared by
        // cross-multiplying (the counts are positive).
        const double ssum = (j < w) ? wsum : ns.step_sum;
        const int sn = (j < w) ? wn : j + 1;
        bool above;                                   // H >= tau (then T_high)
        if (p.threshold == RESET_THRESHOLD_FIXED) {
          above = !(H < (double)p.tau0);
        } else if (p.threshold == RESET_THRESHOLD_WINDOW) {
          above = !(H * wn < wsum);
        } else {
          const bool confident = ssum * t1 <= ns.glob_sum * sn;   // H_step <= H_bar
          above = confident ? !(H < (double)p.tau0) : !(H * sn < ssum);
        }
        low = !above;
      }
      const float T = low ? p.t_low : p.t_high;
      if (rank == 0) {
        if (!state_ok) atomicOr(&g_nvfp4_device_error, NVFP4_DEVERR_STATE_W);
        if (state_ok) {
          RowState* stw = reinterpret_cast<RowState*>(state + (size_t)row * stride);
          reinterpret_cast<double*>(stw + 1)[ns.t % w] = H;
          stw->glob_sum = ns.glob_sum;
          stw->step_sum = ns.step_sum;
          stw->t = t1;
          stw->j = j + 1;
        }
        if (H_out) H_out[row] = (float)H;
        if (T_out) T_out[row] = T;
      }
    }
    low = __shfl_sync(0xffffffffu, low, 0);
    // The CTA that holds u * Z_T: the first whose running total passes the
    // target, else the last CTA with mass.  The target within it is in its
    // own units (relative to its maximum), as its per-warp and per-thread
    // sums are.
    const float zr = low ? zlr : zhr;
    const float target = __ldg(u + row) * (low ? ztl : zth);
    float zi = zr;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, zi, o);
      if (lane >= o) zi += n;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, has && zi > target);
    const unsigned pos = __ballot_sync(0xffffffffu, zr > 0.0f);
    const int rstar = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    const float before = __shfl_sync(0xffffffffu, zi - zr, rstar);
    const float fsel = __shfl_sync(0xffffffffu, low ? fl : fh, rstar);
    if (lane == 0) {
      s_gm = gmax;
      s_T = low ? p.t_low : p.t_high;
      s_rstar = rstar;
      s_zi = low ? 3 : 4;
      s_tl = fsel > 0.0f ? (target - before) / fsel : 0.0f;   // the target within CTA rstar
    }
  }
  __syncthreads();
  const float gm = s_gm;
  if constexpr (NUC) {                              // top-p (NUC is set iff 0 < top_p < 1)
    const float cT = (s_T == p.t_low) ? cl : ch;
    const int tok =
        cluster_nucleus<PER>(reinterpret_cast<const float*>(s_dyn), i0, hi, gm, cT, p, rank, CS, __ldg(u + row));
    if (tok >= 0 && (threadIdx.x & 31) == 0) token[row] = tok;
    return;
  }
  if ((int)rank != s_rstar) return;

  // ---- the token in this CTA: the warp from the per-warp Z_T sums, the lane
  // from the threads' kept totals, then the lane's own logits ----
  const int zi = s_zi;
  if (warp == 0) {
    const float tl = s_tl;
    const float wt = s_wred[zi][lane];
    float wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    // The first warp whose running total passes the target; else the last
    // warp that holds logits of this CTA.
    const unsigned hit = __ballot_sync(0xffffffffu, wi > tl);
    const int nlive = (hi - lo + 32 * PER - 1) / (32 * PER);
    const int wsel = hit ? __ffs(hit) - 1 : nlive - 1;
    const float wb = __shfl_sync(0xffffffffu, wi - wt, wsel);
    if (lane == 0) {
      s_warp = wsel;
      s_tl = tl - wb;
    }
  }
  __syncthreads();
  if (warp == s_warp) {
    const float tl = s_tl;
    const float mine = (zi == 3) ? my_zl : my_zh;
    float incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > tl);
    const int lsel = hit ? __ffs(hit) - 1 : 31;
    if (lane == lsel) {
      const float cT = (zi == 3) ? cl : ch;
      float run = incl - mine;
      int tok = -1, last = -1;
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        if (i0 + k < hi) {
          run += exp2f((v[k] - mb) * cT);
          last = i0 + k;
          if (run > tl && tok < 0) tok = i0 + k;
        }
      }
      // Rounding can leave the target just past the lane's last partial sum
      // (or the lane may hold no logit): the sample is then the last logit of
      // the warp's range that exists.
      token[row] = tok >= 0 ? tok : (last >= 0 ? last : min(hi, lo + (warp + 1) * 32 * PER) - 1);
    }
  }
}

// ---- top-p launches ---------------------------------------------------------------

// Exclusive scan of one value per thread across the CTA; *total gets the sum.
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long* s_w,
                                                                  unsigned long long* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  unsigned long long base = 0ull, all = 0ull;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) base += s_w[w];
    all += s_w[w];
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// One radix level of the nucleus boundary search.  The boundary key is the
// smallest key whose inclusive mass (over keys <= it) reaches ceil(top_p * Z):
// every logit at or above it is kept.  Level 0 bins the whole row by key bits
// 31..21; level 1 the logits whose bits 31..21 equal the chosen digit, by bits
// 20..10; level 2 those matching bits 31..10, by bits 9..0.  Each CTA bins its
// chunk in shared memory and adds the non-zero bins to the row's histogram;
// the last CTA of the row picks the digit, records it and clears the histogram.
template <int level>
__global__ void __launch_bounds__(kThreads) nucleus_level_kernel(const float* __restrict__ logits, int V, int NC,
                                                                float top_p, float mscale, NucRow* nrows,
                                                                unsigned long long* hist, unsigned int* counters) {
  __shared__ unsigned long long s_h[kHistBins];
  __shared__ unsigned long long s_w[kThreads / 32];
  __shared__ int s_last, s_b;
  const int row = blockIdx.x / NC, c = blockIdx.x % NC;
  const float* base = logits + (size_t)row * V;
  const int lo = c * kChunk, hi = min(V, lo + kChunk);
  NucRow* nr = nrows + row;
  const float gmax = __ldcg(&nr->gmax), T = __ldcg(&nr->T);
  const float invT = 1.0f / T;
  const unsigned int prefix = __ldcg(&nr->prefix);
  constexpr int nb = (level == 2) ? 1024 : kHistBins;
  for (int b = threadIdx.x; b < nb; b += kThreads) s_h[b] = 0ull;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int i = lo + threadIdx.x + k * kThreads;
    if (i < hi) {
      const float l = __ldcg(base + i);
      const uint32_t key = nucleus_key(l);
      bool match;
      uint32_t d;
      if constexpr (level == 0) {
        match = true;
        d = key >> 21;
      } else if constexpr (level == 1) {
        match = (key >> 21) == prefix;
        d = (key >> 10) & 0x7FFu;
      } else {
        match = (key >> 10) == prefix;
        d = key & 0x3FFu;
      }
      if (match) {
        const unsigned long long m = nucleus_mass(l, gmax, invT, mscale);
        if (m) atomicAdd(&s_h[d], m);
      }
    }
  }
  __syncthreads();
  unsigned long long* h = hist + (size_t)row * kHistBins;
  for (int b = threadIdx.x; b < nb; b += kThreads)
    if (s_h[b]) atomicAdd(h + b, s_h[b]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counters + row, 1u) == (unsigned int)(NC - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- last CTA of the row: thread t owns bins [t per, (t+1) per) ----
  constexpr int per = nb / kThreads;   // 8 or 4
  unsigned long long hv[per];
  unsigned long long tsum = 0ull;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    hv[j] = __ldcg(h + threadIdx.x * per + j);
    tsum += hv[j];
  }
  unsigned long long total;
  const unsigned long long excl = block_excl_scan_u64(tsum, s_w, &total);
  unsigned long long below, target;
  if constexpr (level == 0) {
    // total >= 1: the maximum's mass is mscale.
    const double t = ceil((double)top_p * (double)total);
    target = (unsigned long long)t;
    if (target < 1ull) target = 1ull;
    if (target > total) target = total;
    below = 0ull;
  } else {
    below = __ldcg(&nr->below);
    target = __ldcg(&nr->target);
  }
  if (threadIdx.x == 0) s_b = 0x7fffffff;
  __syncthreads();
  {
    unsigned long long run = below + excl;
    int first = -1;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      if (first < 0 && run + hv[j] >= target) first = j;
      run += hv[j];
    }
    if (first >= 0) atomicMin(&s_b, threadIdx.x * per + first);
  }
  __syncthreads();
  int b = s_b;
  // The masses of every level are the same integers, so the range chosen at
  // the level before always reaches the target; the fallback is unreachable.
  if (b == 0x7fffffff) b = nb - 1;
  if (threadIdx.x == b / per) {
    unsigned long long nb_below = below + excl;
#pragma unroll
    for (int j = 0; j < per; ++j)
      if (j < b % per) nb_below += hv[j];
    nr->below = nb_below;
    if constexpr (level == 0) {
      nr->target = target;
      nr->prefix = (unsigned int)b;
    } else if constexpr (level == 1) {
      nr->prefix = (prefix << 11) | (unsigned int)b;
    } else {
      nr->prefix = (prefix << 10) | (unsigned int)b;
      unsigned long long hb = 0ull;
#pragma unroll
      for (int j = 0; j < per; ++j)
        if (j == b % per) hb = hv[j];
      nr->zk = nb_below + hb;
    }
  }
#pragma unroll
  for (int j = 0; j < per; ++j) h[threadIdx.x * per + j] = 0ull;   // ready for the next level or call
  if (threadIdx.x == 0) counters[row] = 0u;
}

// Kept mass of each chunk, then (last CTA of the row) the inverse-CDF sample
// over the kept logits: the first chunk whose running sum passes u * Zk, and a
// prefix scan of that one chunk -- all in exact integers.
__global__ void __launch_bounds__(kThreads) nucleus_sample_kernel(const float* __restrict__ logits, int V, int NC,
                                                                 const float* __restrict__ u, float mscale,
                                                                 const NucRow* nrows, unsigned long long* csum,
                                                                 unsigned int* counters, int32_t* token) {
  __shared__ unsigned long long s_w[kThreads / 32];
  __shared__ unsigned long long s_target;
  __shared__ int s_last, s_chunk, s_tok;
  const int row = blockIdx.x / NC, c = blockIdx.x % NC;
  const float* base = logits + (size_t)row * V;
  const int lo = c * kChunk, hi = min(V, lo + kChunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const NucRow* nr = nrows + row;
  const float gmax = __ldcg(&nr->gmax), T = __ldcg(&nr->T);
  const float invT = 1.0f / T;
  const unsigned int kstar = __ldcg(&nr->prefix);

  unsigned long long ms = 0ull;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const int i = lo + threadIdx.x + k * kThreads;
    if (i < hi) {
      const float l = __ldcg(base + i);
      if (nucleus_key(l) <= kstar) ms += nucleus_mass(l, gmax, invT, mscale);
    }
  }
  ms = warp_sum_u64(ms);
  if (lane == 0) s_w[warp] = ms;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0ull;
    for (int w = 0; w < kThreads / 32; ++w) t += s_w[w];
    __stcg(csum + (size_t)row * NC + c, t);
    __threadfence();
    s_last = (atomicAdd(counters + row, 1u) == (unsigned int)(NC - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const unsigned long long* crow = csum + (size_t)row * NC;
  if (warp == 0) {
    const int per = (NC + 31) / 32;
    const int q0 = lane * per, q1 = min(NC, q0 + per);
    unsigned long long mine = 0ull;
    for (int q = q0; q < q1; ++q) mine += __ldcg(crow + q);
    unsigned long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
    // token = min{ i : P_i > u * Zk } with integer prefix sums P: P > u Zk <=> P > floor(u Zk)
    unsigned long long tgt = (unsigned long long)floor((double)__ldg(u + row) * (double)total);
    if (tgt >= total) tgt = total - 1ull;
    const unsigned hit = __ballot_sync(0xffffffffu, q0 < q1 && incl > tgt);
    const int owner = hit ? __ffs(hit) - 1 : (NC - 1) / per;
    if (lane == owner) {
      unsigned long long before = incl - mine;
      int cstar = q1 - 1;
      for (int q = q0; q < q1; ++q) {
        const unsigned long long v = __ldcg(crow + q);
        if (before + v > tgt) {
          cstar = q;
          break;
        }
        before += v;
      }
      s_chunk = cstar;
      s_target = tgt - before;
      s_tok = 0x7fffffff;
    }
  }
  __syncthreads();
  const int clo = s_chunk * kChunk;
  const int chi = min(V, clo + kChunk);
  const int i0 = clo + threadIdx.x * kPerThread;
  float lv[kPerThread];
  if ((V & 3) == 0 && i0 + kPerThread <= chi) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(base + i0));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(base + i0) + 1);
    lv[0] = a.x; lv[1] = a.y; lv[2] = a.z; lv[3] = a.w;
    lv[4] = b.x; lv[5] = b.y; lv[6] = b.z; lv[7] = b.w;
  } else {
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) lv[k] = (i0 + k < chi) ? __ldcg(base + i0 + k) : 0.0f;
  }
  unsigned long long pre[kPerThread];
  unsigned long long run = 0ull;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    if (i0 + k < chi && nucleus_key(lv[k]) <= kstar) run += nucleus_mass(lv[k], gmax, invT, mscale);
    pre[k] = run;
  }
  unsigned long long total;
  const unsigned long long excl = block_excl_scan_u64(run, s_w, &total);
  const unsigned long long target = s_target;
  int cand = 0x7fffffff;
#pragma unroll
  for (int k = kPerThread - 1; k >= 0; --k) {
    if (i0 + k < chi && excl + pre[k] > target) cand = i0 + k;
  }
  if (cand != 0x7fffffff) atomicMin(&s_tok, cand);
  __syncthreads();
  if (threadIdx.x == 0) {
    // Exact sums always find the token; the fallback is unreachable.
    token[row] = (s_tok != 0x7fffffff) ? s_tok : (chi - 1);
    counters[row] = 0u;
  }
}

__global__ void reset_state_init_kernel(uint8_t* state, int M, int w, int stride) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= M) return;
  RowState* st = reinterpret_cast<RowState*>(state + (size_t)r * stride);
  st->t = 0;
  st->j = 0;
  st->w = w;
  st->pad = 0;
  st->glob_sum = 0.0;
  st->step_sum = 0.0;
  double* ring = reinterpret_cast<double*>(st + 1);
  for (int i = 0; i < w; ++i) ring[i] = 0.0;
}

// Row counters first, at a fixed place for every M, so one zeroed workspace
// serves calls of any shape.  Nothing else in the scratch needs to start
// zeroed: the first launch clears a row's histogram before the top-p launches
// add to it.
constexpr size_t kCounterBytes = 256;   // kMaxRows counters

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct SampleLayout {
  size_t parts, nrows, hist, csum, total;
};

SampleLayout sample_layout(int M, int NC) {
  SampleLayout L;
  L.parts = kCounterBytes;
  L.nrows = align256(L.parts + (size_t)M * NC * sizeof(Part));
  L.hist = align256(L.nrows + (size_t)M * sizeof(NucRow));
  L.csum = L.hist + (size_t)M * kHistBins * sizeof(unsigned long long);
  L.total = L.csum + (size_t)M * NC * sizeof(unsigned long long);
  return L;
}

// 2^(62 - ceil(log2 V)): V masses of at most this value sum below 2^63.
float mass_scale(int V) {
  int lg = 0;
  while ((1ll << lg) < (long long)V) ++lg;
  return ldexpf(1.0f, 62 - lg);
}

}  // namespace

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);
nvfp4_status nvfp4_internal_check_device();

namespace {

nvfp4_status check_params(const reset_params* p) {
  if (!(p->t_low > 0.0f) || !(p->t_high > 0.0f) || p->w < 1 || p->w > kMaxW || !(p->tau0 == p->tau0))
    return NVFP4_ERR_RANGE;
  if (p->t_low == p->t_high) return NVFP4_ERR_RANGE;   // the two branches must be distinguishable
  if (p->threshold < RESET_THRESHOLD_RESET || p->threshold > RESET_THRESHOLD_WINDOW) return NVFP4_ERR_RANGE;
  if (!(p->top_p >= 0.0f && p->top_p <= 1.0f)) return NVFP4_ERR_RANGE;   // NaN fails too
  return NVFP4_OK;
}

// The cluster sampler for V logits per row: PER logits per thread (12, 20 or
// 32) and CS <= 8 CTAs per row; false when V needs more (the multi-launch
// path then serves).
template <int PER, bool NUC>
nvfp4_status launch_cluster_per(const float* logits, int M, int V, int CS, const uint8_t* step_start, const float* u,
                                void* state, const Params& prm, int32_t* token, float* H_out, float* T_out,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(M * CS));
  cfg.blockDim = dim3(kCThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (NUC) {
    // top-p keeps each logit's 2^a mscale and rank 0's gathered logits in
    // dynamic shared memory, above the default 48 KB: granted once per device
    const int bytes = (int)cluster_nucleus_smem<PER>();
    static PerDeviceInt granted;
    cudaError_t err = cudaSuccess;
    granted.get(
        [&](int, cudaError_t* e) {
          *e = cudaFuncSetAttribute(reset_cluster_kernel<PER, NUC>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
          return *e == cudaSuccess ? 1 : 0;
        },
        &err);
    if (err != cudaSuccess) return nvfp4_internal_cuda_status(err);
    cfg.dynamicSmemBytes = (size_t)bytes;
  }
  return nvfp4_internal_cuda_status(cudaLaunchKernelEx(&cfg, reset_cluster_kernel<PER, NUC>, logits, V, CS, step_start, u,
                                                       static_cast<uint8_t*>(state), (int)state_stride(prm.w), prm,
                                                       token, H_out, T_out));
}

template <bool NUC>
bool launch_cluster_nuc(const float* logits, int M, int V, const uint8_t* step_start, const float* u, void* state,
                        const Params& prm, int32_t* token, float* H_out, float* T_out, cudaStream_t stream,
                        nvfp4_status* st) {
  const long long per_cta12 = (long long)kCThreads * 12, per_cta20 = (long long)kCThreads * 20,
                  per_cta32 = (long long)kCThreads * 32;
  if (V <= kMaxClusterCtas * per_cta12) {
    *st = launch_cluster_per<12, NUC>(logits, M, V, (int)((V + per_cta12 - 1) / per_cta12), step_start, u, state,
                                      prm, token, H_out, T_out, stream);
  } else if (V <= kMaxClusterCtas * per_cta20) {
    *st = launch_cluster_per<20, NUC>(logits, M, V, (int)((V + per_cta20 - 1) / per_cta20), step_start, u, state,
                                      prm, token, H_out, T_out, stream);
  } else if (V <= kMaxClusterCtas * per_cta32) {
    *st = launch_cluster_per<32, NUC>(logits, M, V, (int)((V + per_cta32 - 1) / per_cta32), step_start, u, state,
                                      prm, token, H_out, T_out, stream);
  } else {
    return false;
  }
  return true;
}

// The cluster sampler when the row fits one cluster (V <= 8 x 1024 x 32);
// false otherwise (the multi-launch path then serves).
bool launch_cluster(const float* logits, int M, int V, const uint8_t* step_start, const float* u, void* state,
                    const Params& prm, int32_t* token, float* H_out, float* T_out, cudaStream_t stream,
                    nvfp4_status* st) {
  const bool nuc = prm.top_p > 0.0f && prm.top_p < 1.0f;
  return nuc ? launch_cluster_nuc<true>(logits, M, V, step_start, u, state, prm, token, H_out, T_out, stream, st)
             : launch_cluster_nuc<false>(logits, M, V, step_start, u, state, prm, token, H_out, T_out, stream, st);
}

// The sampler's launches for M rows in `scratch` (laid out by sample_layout).
nvfp4_status launch_sample(const float* logits, int M, int V, int NC, const uint8_t* step_start, const float* u,
                           void* state, const reset_params* p, int32_t* token, float* H_out, float* T_out,
                           uint8_t* scratch, cudaStream_t stream) {
  const SampleLayout L = sample_layout(M, NC);
  unsigned int* counters = reinterpret_cast<unsigned int*>(scratch);
  Part* parts = reinterpret_cast<Part*>(scratch + L.parts);
  NucRow* nrows = reinterpret_cast<NucRow*>(scratch + L.nrows);
  unsigned long long* hist = reinterpret_cast<unsigned long long*>(scratch + L.hist);
  unsigned long long* csum = reinterpret_cast<unsigned long long*>(scratch + L.csum);
  const bool nucleus = p->top_p > 0.0f && p->top_p < 1.0f;
  Params prm{p->tau0, p->t_low, p->t_high, p->w, p->threshold, p->top_p, mass_scale(V)};
  {
    nvfp4_status cst = NVFP4_OK;
    if (launch_cluster(logits, M, V, step_start, u, state, prm, token, H_out, T_out, stream, &cst)) return cst;
  }
  reset_sample_kernel<<<M * NC, kThreads, 0, stream>>>(logits, M, V, NC, step_start, u, static_cast<uint8_t*>(state),
                                                        (int)state_stride(p->w), prm, token, H_out, T_out, parts,
                                                        counters, nucleus ? nrows : nullptr, hist);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !nucleus) return nvfp4_internal_cuda_status(e);
  const float mscale = mass_scale(V);
  nucleus_level_kernel<0><<<M * NC, kThreads, 0, stream>>>(logits, V, NC, p->top_p, mscale, nrows, hist, counters);
  nucleus_level_kernel<1><<<M * NC, kThreads, 0, stream>>>(logits, V, NC, p->top_p, mscale, nrows, hist, counters);
  nucleus_level_kernel<2><<<M * NC, kThreads, 0, stream>>>(logits, V, NC, p->top_p, mscale, nrows, hist, counters);
  e = cudaGetLastError();
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  nucleus_sample_kernel<<<M * NC, kThreads, 0, stream>>>(logits, V, NC, u, mscale, nrows, csum, counters, token);
  return nvfp4_internal_cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" size_t reset_state_bytes(int M, int w) {
  if (M < 1 || M > kMaxRows || w < 1 || w > kMaxW) return 0;
  return (size_t)M * state_stride(w);
}

extern "C" nvfp4_status reset_state_init(void* state, int M, int w, cudaStream_t stream) {
  if (!state) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxRows || w < 1 || w > kMaxW) return NVFP4_ERR_RANGE;
  if (!nvfp4_internal_aligned(state, 16)) return NVFP4_ERR_ALIGN;
  reset_state_init_kernel<<<1, kMaxRows, 0, stream>>>(static_cast<uint8_t*>(state), M, w, (int)state_stride(w));
  return nvfp4_internal_cuda_status(cudaGetLastError());
}

extern "C" size_t reset_workspace_bytes(int M, int V) {
  if (M < 1 || M > kMaxRows || V < 1 || V > (1 << 24)) return 0;
  const int NC = (V + kChunk - 1) / kChunk;
  return sample_layout(M, NC).total;
}

extern "C" nvfp4_status reset_sample(const float* logits, int M, int V, const uint8_t* step_start, const float* u,
                                     void* state, const reset_params* p, int32_t* token, float* H_out, float* T_out,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!logits || !u || !state || !p || !token || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxRows) return NVFP4_ERR_RANGE;
  if (V < 1 || V > (1 << 24)) return NVFP4_ERR_SHAPE;
  nvfp4_status ps = check_params(p);
  if (ps != NVFP4_OK) return ps;
  if (!nvfp4_internal_aligned(logits, 16) || !nvfp4_internal_aligned(state, 16) ||
      !nvfp4_internal_aligned(workspace, 256) || !nvfp4_internal_aligned(u, 4) || !nvfp4_internal_aligned(token, 4))
    return NVFP4_ERR_ALIGN;
  const int NC = (V + kChunk - 1) / kChunk;
  if (NC > 1024) return NVFP4_ERR_SHAPE;
  if (workspace_bytes < reset_workspace_bytes(M, V)) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  return launch_sample(logits, M, V, NC, step_start, u, state, p, token, H_out, T_out,
                       static_cast<uint8_t*>(workspace), stream);
}

// ---- allocation-free variant ------------------------------------------------------
// Same launches, with their scratch (row counters, per-chunk partials, the
// top-p records and histograms) in a file-scope device array instead of a
// caller workspace, for callers that may not allocate device memory.  The
// array is reserved on every GPU that loads the library, until the process
// exits.
namespace {
constexpr int kNoAllocMaxChunks = 4096;   // limit on M * ceil(V / 2048)
constexpr size_t kNoAllocScratchBytes =
    kCounterBytes + (size_t)kNoAllocMaxChunks * (sizeof(Part) + sizeof(unsigned long long)) +
    (size_t)kMaxRows * (sizeof(NucRow) + kHistBins * sizeof(unsigned long long)) + 512;   // 1,217,280
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
uint8_t* g_noalloc_scratch_dev[kNoAllocMaxDevices] = {};
}  // namespace

static __device__ __align__(256) uint8_t g_reset_noalloc_scratch[kNoAllocScratchBytes];

// Device address of this device's copy of the array (host code may not use the
// array's name as a device pointer).  Looked up once per device.
static cudaError_t noalloc_scratch_address(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_reset_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_scratch_dev[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_scratch_dev[dev];
  return cudaSuccess;
}

extern "C" nvfp4_status reset_sample_noalloc(const float* logits, int M, int V, const uint8_t* step_start,
                                             const float* u, void* state, const reset_params* p, int32_t* token,
                                             float* H_out, float* T_out, cudaStream_t stream) {
  if (!logits || !u || !state || !p || !token) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxRows) return NVFP4_ERR_RANGE;
  if (V < 1 || V > (1 << 24)) return NVFP4_ERR_SHAPE;
  nvfp4_status ps = check_params(p);
  if (ps != NVFP4_OK) return ps;
  if (!nvfp4_internal_aligned(logits, 16) || !nvfp4_internal_aligned(state, 16) || !nvfp4_internal_aligned(u, 4) ||
      !nvfp4_internal_aligned(token, 4))
    return NVFP4_ERR_ALIGN;
  const int NC = (V + kChunk - 1) / kChunk;
  // Rows of up to 8 x 1024 x 32 logits take one cluster a row and use no
  // scratch; longer rows take the multi-launch path and its static array.
  const bool one_cluster = V <= kMaxClusterCtas * kCThreads * 32;
  if (!one_cluster) {
    if (NC > 1024 || (long long)M * NC > kNoAllocMaxChunks) return NVFP4_ERR_SHAPE;   // beyond the static scratch
    if (sample_layout(M, NC).total > kNoAllocScratchBytes) return NVFP4_ERR_SHAPE;
  }
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  uint8_t* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  if (!one_cluster) {
    // The array keeps the previous call's contents: clear the row counters.
    e = cudaMemsetAsync(scratch, 0, kCounterBytes, stream);
    if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  }
  return launch_sample(logits, M, V, NC, step_start, u, state, p, token, H_out, T_out, scratch, stream);
}
