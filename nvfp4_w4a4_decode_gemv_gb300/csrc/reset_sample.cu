// ReSET step-aware temperature sampler (one decode position, M rows).
//
// Rule (ReSET project page, "Step-aware temperature scaling"; reading note
// §3.1 Eq. (1), §3.2, §4.1 SAT, §4.2 HSE, §4.3):
//   H      = entropy of softmax(logits)            (nats, temperature 1)
//   H_step = mean of the last w entropies while the in-step position j < w,
//            else the running mean of the step's entropies
//   H_bar  = running mean of all entropies of the sequence
//   tau    = tau0 if H_step <= H_bar (confident step) else H_step
//   T      = T_low if H < tau else T_high
//   token  = min{ i : sum_{k<=i} p_k > u * sum_k p_k },  p_k = exp((l_k - max l) / T)
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
};

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
                                                               float* T_out, Part* parts, unsigned int* counters) {
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
        a1 += e * s;
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
      if (!state_ok) atomicExch(&g_nvfp4_device_error, NVFP4_DEVERR_STATE_W);
      double Hs = 0.0, Hbar = 0.0;
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
        if (j < w) {
          if (t1 <= w) {
            Hs = st->glob_sum / t1;             // the window is the whole history
          } else {
            double ws = 0.0;
            for (int i = 0; i < w; ++i) ws += ring[i];
            Hs = ws / w;
          }
        } else {
          Hs = st->step_sum / (j + 1);
        }
        Hbar = st->glob_sum / t1;
      }
      const double tau = (Hs <= Hbar) ? (double)p.tau0 : Hs;
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
// serves calls of any shape.
constexpr size_t kCounterBytes = 256;   // kMaxRows counters

}  // namespace

nvfp4_status nvfp4_internal_cuda_status(cudaError_t e);
bool nvfp4_internal_aligned(const void* p, size_t a);
nvfp4_status nvfp4_internal_check_device();

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
  return kCounterBytes + (size_t)M * NC * sizeof(Part);
}

extern "C" nvfp4_status reset_sample(const float* logits, int M, int V, const uint8_t* step_start, const float* u,
                                     void* state, const reset_params* p, int32_t* token, float* H_out, float* T_out,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!logits || !u || !state || !p || !token || !workspace) return NVFP4_ERR_NULL;
  if (M < 1 || M > kMaxRows) return NVFP4_ERR_RANGE;
  if (V < 1 || V > (1 << 24)) return NVFP4_ERR_SHAPE;
  if (!(p->t_low > 0.0f) || !(p->t_high > 0.0f) || p->w < 1 || p->w > kMaxW || !(p->tau0 == p->tau0))
    return NVFP4_ERR_RANGE;
  if (p->t_low == p->t_high) return NVFP4_ERR_RANGE;   // the two branches must be distinguishable
  if (!nvfp4_internal_aligned(logits, 16) || !nvfp4_internal_aligned(state, 16) ||
      !nvfp4_internal_aligned(workspace, 256) || !nvfp4_internal_aligned(u, 4) || !nvfp4_internal_aligned(token, 4))
    return NVFP4_ERR_ALIGN;
  const int NC = (V + kChunk - 1) / kChunk;
  if (NC > 1024) return NVFP4_ERR_SHAPE;
  if (workspace_bytes < reset_workspace_bytes(M, V)) return NVFP4_ERR_SHAPE;
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  Params prm{p->tau0, p->t_low, p->t_high, p->w};
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  unsigned int* counters = reinterpret_cast<unsigned int*>(wsb);
  Part* parts = reinterpret_cast<Part*>(wsb + kCounterBytes);
  reset_sample_kernel<<<M * NC, kThreads, 0, stream>>>(logits, M, V, NC, step_start, u, static_cast<uint8_t*>(state),
                                                        (int)state_stride(p->w), prm, token, H_out, T_out, parts,
                                                        counters);
  return nvfp4_internal_cuda_status(cudaGetLastError());
}

// ---- allocation-free variant ------------------------------------------------------
// Same kernel, with its scratch (row counters, then per-chunk partials) in a
// file-scope device array instead of a caller workspace, for callers that may
// not allocate device memory.  The array is reserved on every GPU that loads
// the library, until the process exits.
namespace {
constexpr int kNoAllocMaxChunks = 4096;   // limit on M * ceil(V / 2048)
constexpr size_t kNoAllocScratchBytes = kCounterBytes + (size_t)kNoAllocMaxChunks * sizeof(Part);   // 131,328
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
  if (!(p->t_low > 0.0f) || !(p->t_high > 0.0f) || p->w < 1 || p->w > kMaxW || !(p->tau0 == p->tau0))
    return NVFP4_ERR_RANGE;
  if (p->t_low == p->t_high) return NVFP4_ERR_RANGE;
  if (!nvfp4_internal_aligned(logits, 16) || !nvfp4_internal_aligned(state, 16) || !nvfp4_internal_aligned(u, 4) ||
      !nvfp4_internal_aligned(token, 4))
    return NVFP4_ERR_ALIGN;
  const int NC = (V + kChunk - 1) / kChunk;
  if (NC > 1024 || (long long)M * NC > kNoAllocMaxChunks) return NVFP4_ERR_SHAPE;   // beyond the static scratch
  nvfp4_status ds = nvfp4_internal_check_device();
  if (ds != NVFP4_OK) return ds;
  uint8_t* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  // The array keeps the previous call's contents: clear the row counters.
  e = cudaMemsetAsync(scratch, 0, kCounterBytes, stream);
  if (e != cudaSuccess) return nvfp4_internal_cuda_status(e);
  Params prm{p->tau0, p->t_low, p->t_high, p->w};
  reset_sample_kernel<<<M * NC, kThreads, 0, stream>>>(logits, M, V, NC, step_start, u, static_cast<uint8_t*>(state),
                                                        (int)state_stride(p->w), prm, token, H_out, T_out,
                                                        reinterpret_cast<Part*>(scratch + kCounterBytes),
                                                        reinterpret_cast<unsigned int*>(scratch));
  return nvfp4_internal_cuda_status(cudaGetLastError());
}
