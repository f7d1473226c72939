/*
 * nvfp4.h -- C ABI of the NVFP4 W4A4 small-M decode library for GB300 (sm_103a).
 *
 * What it computes (the ReSET pages):
 *   - NVFP4 = E2M1 4-bit elements, one E4M3 scale per 16 consecutive elements
 *     along K, one FP32 global scale per tensor (ReSET reading note, §2.1;
 *     §6.1 setup: "E2M1 elements, E4M3 block scales, group size 16").
 *   - The small-M decode projection Y = dequant(Xq) . dequant(Wq)^T for
 *     M = 1..8 active tokens, computed without a 128-row tensor-core tile
 *     (ReSET project page, "Why a CUDA-core NVFP4 kernel?" and "Core
 *     contribution -- the nvfp4r CUDA-core kernel", design choices C1-C3).
 *   - The ReSET step-aware temperature sampler: token entropy, online step
 *     entropy estimate (HSE), step-aware threshold (SAT), two-temperature
 *     sample (project page, "Step-aware temperature scaling"; reading note
 *     §3.1, §4.1-§4.3).
 *
 * Conventions for every entry point:
 *   - Data pointers are DEVICE pointers owned by the caller; the library keeps
 *     no reference after the call returns and allocates nothing.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *     may be captured into a CUDA graph, except where a function says otherwise.
 *   - Argument errors are reported synchronously, before anything is launched:
 *     NVFP4_ERR_NULL, NVFP4_ERR_SHAPE, NVFP4_ERR_ALIGN, NVFP4_ERR_RANGE.
 *     A failed launch returns NVFP4_ERR_CUDA; nvfp4_last_cuda_error() names it.
 *   - Tensors are row-major and dense.  NVFP4 tensor layout:
 *       codes  uint8 [rows, K/2]  element 2j in the low nibble of byte j,
 *                                 element 2j+1 in the high nibble;
 *       scales uint8 [rows, K/16] E4M3 (OCP "fn") scale of elements 16b..16b+15,
 *                                 not interleaved;
 *       global float (one, on the device) -- dequant: x = e2m1(c) * e4m3(s) * global.
 *   - Calls on distinct streams are independent, except where a function
 *     says that concurrent calls share a buffer.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,   /* a required pointer is NULL */
  NVFP4_ERR_SHAPE = 2,  /* a size is negative, too large or not a required multiple */
  NVFP4_ERR_ALIGN = 3,  /* a pointer is not aligned as the function requires */
  NVFP4_ERR_RANGE = 4,  /* a parameter value is out of range (M, temperatures, w, ...) */
  NVFP4_ERR_CUDA = 5,   /* a CUDA runtime call or a kernel launch failed */
  NVFP4_ERR_DEVICE = 6  /* the current device is not a Blackwell sm_100-family GPU */
} nvfp4_status;

/* Static string for a status code. */
const char* nvfp4_status_str(nvfp4_status s);

/* Text of the last CUDA error seen by this library in the calling thread (static storage). */
const char* nvfp4_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
int nvfp4_version(void);

/*
 * Reads and clears the device error bits of the current device (the OR of
 * every error any kernel recorded since the last read).  A kernel sets a bit
 * when one of its bounded waits gave up, then returns early with incomplete
 * outputs:
 *   bit 0 (1)  a wait on an mbarrier (a TMA copy or an MMA that never completed);
 *   bit 1 (2)  reset_sample called with a state built for a smaller window;
 *   bit 2 (4)  a GEMV CTA's wait for another CTA's partial sum.  After this
 *              error the GEMV workspace may hold a partial sum published after
 *              the wait gave up: zero the workspace again before its next use.
 * Synchronous (it copies a few bytes from the device); not for use inside
 * stream capture.
 */
nvfp4_status nvfp4_device_status(unsigned int* code);

/* ------------------------------------------------------------------------ */
/* Quantizer: BF16 -> NVFP4                                                   */
/* ------------------------------------------------------------------------ */
/*
 * Quantizes x[rows, K] (BF16 bit patterns) by the NVFP4 two-level recipe, all
 * in FP32 with IEEE rounding at each step:
 *   amax = max|x| over the whole tensor; global = amax / 2688 (448 * 6);
 *   per 16-element block: s = E4M3_rne_satfinite(max|x_block| / (6 * global));
 *   per element: code = E2M1_rne_satfinite(x / (e4m3(s) * global)).
 * The sign bit of each code is the sign bit of x (a negative value that rounds
 * to zero gives 0x8).  When e4m3(s) * global is 0 (all-zero block, a scale that
 * underflows, all-zero tensor) the code is the sign bit alone.
 * Format: ReSET reading note §2.1 and §6.1; the pages' activation quantizer
 * "Q" with a non-interleaved scale layout: reading note §5.3 (Table 3).
 *
 *   x_bf16   device, [rows, K] BF16, 16-byte aligned
 *   rows     >= 0 (activations: the M tokens; weights: N output channels)
 *   K        >= 0, multiple of 16
 *   codes    device, [rows, K/2], 16-byte aligned            (written)
 *   scales   device, [rows, K/16], 4-byte aligned            (written)
 *   global   device, one float, 4-byte aligned               (written)
 * Inputs with NaN or Inf are outside the contract (results unspecified).
 * rows == 0 or K == 0 writes global = 0.
 */
nvfp4_status nvfp4_quantize_act(const uint16_t* x_bf16, int rows, int K, uint8_t* codes,
                                uint8_t* scales, float* global_scale, cudaStream_t stream);

/*
 * Same recipe on FP32 input rows that are first rounded to BF16 (RNE): the
 * values quantized are exactly those nvfp4_quantize_act would see after a
 * FP32->BF16 cast.  Row r of the input starts at x + r * ld (ld >= K, in
 * floats), so a column slice [0, K) of a wider matrix can be quantized in
 * place (the decode step feeds the query columns of the qkv output to the o
 * projection this way).  x 16-byte aligned, ld a multiple of 4.
 */
nvfp4_status nvfp4_quantize_f32(const float* x, int rows, int K, int ld, uint8_t* codes,
                                uint8_t* scales, float* global_scale, cudaStream_t stream);

/*
 * SiLU(gate) * up on FP32 gate_up[rows, 2*I] (gate = columns [0, I), up =
 * columns [I, 2I)), each product computed in FP32 and rounded to BF16, then
 * quantized by the recipe above into codes[rows, I/2], scales[rows, I/16].
 * I a multiple of 16; gate_up 16-byte aligned.  (The MLP of the decode step
 * between the gate_up and down projections.)
 */
nvfp4_status nvfp4_silu_mul_quantize(const float* gate_up, int rows, int I, uint8_t* codes,
                                     uint8_t* scales, float* global_scale, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Small-M NVFP4 GEMV                                                         */
/* ------------------------------------------------------------------------ */
/*
 * y[m, n] = xg * wg * sum_k e2m1(xq[m,k]) e4m3(xs[m,k/16]) e2m1(wq[n,k]) e4m3(ws[n,k/16])
 * for m < M, n < N: the decode projection Y = X W^T of the ReSET project page
 * ("Core contribution": one CTA group reuses each streamed weight tile for all
 * M tokens, several accumulator chains per thread, register-only dequant).
 * Accumulation is FP32 across blocks; the result is within
 * 1e-3 * sum_k |x_k w_k| + 1e-6 of the exact product.
 *
 *   xq, xs, xg   activations in NVFP4 layout, [M, K/2], [M, K/16], one float
 *   M            1..8
 *   wq, ws, wg   weights in NVFP4 layout, [N, K/2], [N, K/16], one float
 *   N            1 .. 2^20
 *   K            >= 256, multiple of 256
 *   y            device, [M, N] FP32 (written)
 *   workspace    device scratch of at least nvfp4_gemv_workspace_bytes(M, N, K)
 *                bytes, 256-byte aligned, ZEROED ONCE before its first use
 *                (cudaMemset); every call leaves it ready for the next one,
 *                whatever the shape of the next call -- unless the call
 *                recorded device error bit 2 (nvfp4_device_status): zero it
 *                again then.
 *                Calls that overlap in time on the GPU must use different
 *                workspaces.
 * Co-residency: the kernel's CTAs (two per SM, one grid of up to 2 x the SM
 * count) exchange partial sums and wait for one another, so all of them must
 * be resident at once.  That holds when the call has the GPU to itself or
 * shares it with other kernels that finish; under MPS limits or green contexts
 * that cap the SMs a context may use, or beside a kernel that never ends, a
 * CTA's wait can run out: the call then records bit 2 and its y is wrong.
 * Alignment: xq, wq, xs, ws 16-byte aligned; y 16-byte aligned.
 */
size_t nvfp4_gemv_workspace_bytes(int M, int N, int K);

nvfp4_status nvfp4_gemv_smallm(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                               const uint8_t* wq, const uint8_t* ws, const float* wg, int N, int K,
                               float* y, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * nvfp4_gemv_smallm computed by a second, independent kernel on the CUDA cores:
 * the pages' own design (ReSET project page, "Core contribution -- the nvfp4r
 * CUDA-core kernel": each weight tile streamed once for all M tokens (C1),
 * several FP32 accumulator chains per thread (C2), dequantization in
 * registers (C3)), with each 16-element block summed exactly in integers.
 * Same arguments, result tolerance, workspace and errors as
 * nvfp4_gemv_smallm; not the fast path (the tensor-core kernel is), kept so
 * that two implementations can be checked against each other.
 */
nvfp4_status nvfp4_gemv_smallm_cudacore(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                        const uint8_t* wq, const uint8_t* ws, const float* wg, int N, int K,
                                        float* y, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/*
 * Test hook for the tensor-core GEMV's bounded wait (no counterpart in the
 * pages).  For every later tensor-core GEMV launch in the process:
 * flag_spin_limit = how many times a CTA polls another CTA's partial sum
 * before giving up (0 = the default, about 2^24 polls), and drop_records != 0
 * makes every CTA skip publishing its partial sums, so that the CTA finishing
 * a split tile waits until the limit, records device error bit 2 and writes a
 * wrong y.  Lets a test make the wait run out without any fault or hang.
 * Call nvfp4_test_gemv_fault(0, 0) to return to normal operation; not
 * thread-safe against concurrent GEMV calls.
 */
void nvfp4_test_gemv_fault(unsigned int flag_spin_limit, int drop_records);

/*
 * Packed weights.  The pages quantize the weights offline, from the BF16
 * checkpoint (ReSET reading note §6.1), and leave their memory layout to the
 * kernel.  nvfp4_pack_weights rewrites wq/ws into blocks of
 * 18432 bytes, one per [128-row tile t] x [256-K chunk c], stored in the order
 * (t, c) with c fastest, so that a GEMV streams each tile chunk as one
 * contiguous read:
 *   bytes [0, 16384)      codes of rows 128t .. 128t+127, K-bytes [128c, 128c+128):
 *                         the 16-byte piece j (0..7) of tile row r (0..127) at
 *                         r*128 + ((j XOR (r mod 8)) * 16)
 *   bytes [16384, 18432)  scales of those rows for blocks [16c, 16c+16): tile
 *                         row r at 16384 + 16 r
 * Rows n >= N of the last tile are zero.  The packed image holds the same
 * bytes as wq and ws (plus the zero rows); nothing is recomputed.
 *
 * nvfp4_packed_weight_bytes(N, K) = ceil(N/128) * (K/256) * 18432, or 0 for an
 * invalid shape (N 1 .. 2^20, K a positive multiple of 256).
 * nvfp4_pack_weights: wq [N, K/2], ws [N, K/16], packed (written) of at least
 * nvfp4_packed_weight_bytes bytes, all device, 16-byte aligned; asynchronous on
 * `stream`; wq/ws must not overlap `packed`.
 * nvfp4_gemv_smallm_packed: nvfp4_gemv_smallm with the weights given packed;
 * same result bits for the same inputs on the tensor-core path, same
 * workspace contract.
 */
size_t nvfp4_packed_weight_bytes(int N, int K);

nvfp4_status nvfp4_pack_weights(const uint8_t* wq, const uint8_t* ws, int N, int K, uint8_t* packed,
                                size_t packed_bytes, cudaStream_t stream);

nvfp4_status nvfp4_gemv_smallm_packed(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                                      const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * nvfp4_quantize_act of a BF16 activation followed by nvfp4_gemv_smallm_packed,
 * as one call: y[m, n] = xg * wg * sum_k e2m1(xq[m,k]) e4m3(xs[m,k/16])
 * e2m1(wq[n,k]) e4m3(ws[n,k/16]), where wq, ws are the codes and scales the
 * packed image holds and xq, xs, xg exactly what nvfp4_quantize_act(x) would
 * write (the
 * activation quantizer "Q" in front of every decode projection: ReSET
 * reading note §5.3, Table 3).  y holds the same bits as the two calls.
 * For M <= 3 and M * K <= 65536 it is one launch (tuning knobs
 * NVFP4_QGEMV_MAX_M, NVFP4_QGEMV_MAX_MK): every CTA of the GEMV reads the
 * whole activation for its maximum and quantizes the 256-K chunks it
 * multiplies into shared memory, so the quantized activation never goes
 * through HBM and one kernel boundary of a decode chain disappears.  Larger
 * activations, or a CTA that would hold more than 24 chunks or quantize more
 * than 1024 blocks (NVFP4_QGEMV_MAX_BLOCKS), take two launches: the library
 * quantizes into the workspace, then multiplies.
 *   x        device, BF16 [M, K] row-major, 16-byte aligned
 *   M        1..8 (else NVFP4_ERR_RANGE)
 *   wpacked, wg, N, K   as nvfp4_gemv_smallm_packed
 *   y        device, [M, N] FP32, 16-byte aligned (written)
 *   xg_out   device float receiving the activation's global scale amax / 2688,
 *            4-byte aligned, or NULL
 *   workspace  device scratch of at least
 *            nvfp4_quantize_gemv_workspace_bytes(M, N, K) bytes, 256-byte
 *            aligned; the same contract as the GEMV workspace (zeroed once,
 *            left ready, one per set of calls that overlap on the GPU); a
 *            zeroed workspace may serve this call and the GEMV calls alike.
 * Errors, co-residency and device error bits as nvfp4_gemv_smallm.
 */
size_t nvfp4_quantize_gemv_workspace_bytes(int M, int N, int K);

/*
 * How nvfp4_quantize_gemv_packed runs a shape on the current device: 1 (one
 * launch), 2 (the quantizer, then the GEMV), 0 for a shape it rejects, -1
 * when the device cannot be queried.  No launch, no synchronization.
 */
int nvfp4_quantize_gemv_launches(int M, int N, int K);

nvfp4_status nvfp4_quantize_gemv_packed(const uint16_t* x_bf16, int M, const uint8_t* wpacked,
                                        const float* wg, int N, int K, float* y, float* xg_out,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Prefill-sized NVFP4 GEMM (M up to 128)                                      */
/* ------------------------------------------------------------------------ */
/*
 * y[m, n] = xg * wg * sum_k e2m1(xq[m,k]) e4m3(xs[m,k/16]) e2m1(w[n,k]) e4m3(sw[n,k/16])
 * for m < M <= 128 and packed weights: the same product as
 * nvfp4_gemv_smallm_packed for a prefill-sized batch of tokens (the pages'
 * own tensor-core GEMM at M = 128: ReSET reading note §7.3, Table 16).  One
 * tcgen05 MMA covers 128 weight rows x 128 tokens x 64 K; each weight block is
 * read from HBM once per call.  FP32 accumulation: within
 * 1e-3 * sum_k |x_k w_k| + 1e-6 of the exact product.
 *   xq, xs, xg   activations, NVFP4 layout [M, K/2], [M, K/16] (16-byte
 *                aligned), one float
 *   M            1..128 (else NVFP4_ERR_RANGE)
 *   wpacked, wg  the weight in the nvfp4_pack_weights layout, one float
 *   N, K         N 1 .. 2^20, K a positive multiple of 256
 *   y            [M, N] FP32, 16-byte aligned (written)
 *   workspace    device scratch of at least nvfp4_gemm_workspace_bytes(M, N, K)
 *                bytes (a fixed size per device: 64 KB per SM), 256-byte
 *                aligned, ZEROED ONCE before its first use and left ready for
 *                the next call of any shape; zero it again after device error
 *                bit 2.  Calls that overlap on the GPU need different workspaces.
 * Co-residency and errors as nvfp4_gemv_smallm.  One CTA per SM.
 */
size_t nvfp4_gemm_workspace_bytes(int M, int N, int K);

nvfp4_status nvfp4_gemm_packed(const uint8_t* xq, const uint8_t* xs, const float* xg, int M,
                               const uint8_t* wpacked, const float* wg, int N, int K, float* y,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* BF16 GEMV (the decode step's lm_head)                                       */
/* ------------------------------------------------------------------------ */
/*
 * y[m, n] = sum_k x[m, k] * w[n, k], BF16 inputs, FP32 accumulation and output.
 * M 1..8, K a multiple of 8 with M * K <= 51200 (x is held in shared memory as
 * FP32), all pointers 16-byte aligned.  Larger M * K returns NVFP4_ERR_SHAPE.
 */
nvfp4_status nvfp4_bf16_gemv(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                             cudaStream_t stream);

/*
 * The same BF16 GEMV on the tensor cores (tcgen05 kind::f16, BF16 x BF16 ->
 * FP32 accumulator in TMEM), on the NVFP4 GEMV's kernel: weight tiles of
 * [128 rows x 64 K] streamed through a shared-memory ring by TMA, Stream-K
 * split over the tiles' K chunks, the same deterministic fix-up.  It needs
 * the records region of a GEMV workspace:
 *   nvfp4_bf16_gemv_workspace_bytes(M, N, K): bytes of workspace needed (0 for
 *   an invalid shape); any buffer that satisfies nvfp4_gemv_workspace_bytes
 *   for the same M also satisfies it, so one zeroed workspace serves both.
 *   x [M, K], w [N, K] BF16 row-major, y [M, N] FP32, all device, 16-byte
 *   aligned; M 1..8, N 1 .. 2^20, K a positive multiple of 64; workspace
 *   256-byte aligned, ZEROED ONCE before its first use, left ready for the
 *   next call.  FP32 accumulation: within 1e-4 * sum_k |x_k w_k| + 1e-6 of
 *   the exact product.  Errors as nvfp4_gemv_smallm.
 */
size_t nvfp4_bf16_gemv_workspace_bytes(int M, int N, int K);

nvfp4_status nvfp4_bf16_gemv_tc(const uint16_t* x, int M, const uint16_t* w, int N, int K, float* y,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * RMS normalization of FP32 rows to BF16 (no gain):
 *   out[r, k] = BF16( x[r, k] / sqrt( (1/K) sum_k x[r, k]^2 + eps ) )
 * Row r of the input starts at x + r * ld (ld >= K, in floats); out is
 * [rows, K] row-major.  The sum of squares is FP32 (in a fixed order per K),
 * the square root and the division IEEE; results are within one BF16 rounding
 * of the exact value.  K a multiple of 4, ld a multiple of 4, x 16-byte and
 * out 8-byte aligned, eps >= 0.
 * The pages' decode step runs inside a Qwen3 decoder, whose layers normalize
 * their inputs (ReSET reading note §6.1: Qwen3 models); the synthetic decode
 * step puts this in front of the qkv and gate_up projections so that a chain
 * of many layers keeps its magnitude (SiLU(gate)*up squares it otherwise).
 */
nvfp4_status nvfp4_rms_norm_bf16(const float* x, int rows, int K, int ld, float eps, uint16_t* out,
                                 cudaStream_t stream);

/*
 * nvfp4_rms_norm_bf16 followed by nvfp4_quantize_act, in one launch: the BF16
 * rows r = BF16(x / sqrt((1/K) sum x^2 + eps)) are quantized by the recipe of
 * nvfp4_quantize_act (one global scale over all rows) into codes [rows, K/2],
 * scales [rows, K/16] and global_scale.  The decode step's normalization in
 * front of the qkv and gate_up projections (see nvfp4_rms_norm_bf16).
 * The row's sum of squares is FP32 in a fixed order (it may differ from
 * nvfp4_rms_norm_bf16's order, so r may differ from that function's output by
 * one BF16 rounding where the exact value is that close to a boundary); the
 * codes are exactly nvfp4_quantize_act of r.  r_out, if not null, receives r
 * ([rows, K] BF16, 16-byte aligned).
 *   rows     0..8 (one CTA per row, the rows forming one thread-block cluster)
 *   K        16..16384, multiple of 16;  ld >= K, multiple of 4 (floats)
 *   eps      >= 0 (a zero row needs eps > 0)
 *   x        device FP32, row r at x + r * ld, 16-byte aligned
 *   codes    16-byte aligned; scales, global_scale 4-byte aligned (written)
 * Errors: NVFP4_ERR_SHAPE (K, ld), NVFP4_ERR_RANGE (rows > 8, eps < 0 or NaN),
 * NVFP4_ERR_NULL, NVFP4_ERR_ALIGN, NVFP4_ERR_CUDA (launch).  rows == 0 writes
 * global_scale = 0.
 */
nvfp4_status nvfp4_rms_norm_quantize(const float* x, int rows, int K, int ld, float eps, uint8_t* codes,
                                     uint8_t* scales, float* global_scale, uint16_t* r_out,
                                     cudaStream_t stream);

/* FP32 -> BF16 (RNE) elementwise cast of n values; x, y 16-byte aligned, n a multiple of 8. */
nvfp4_status nvfp4_f32_to_bf16(const float* x, size_t n, uint16_t* y, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* ReSET sampler                                                              */
/* ------------------------------------------------------------------------ */
/* Threshold policies (reset_params.threshold).  ReSET's own is the default;
 * the other two are the policies the ReSET reading note compares it with
 * (§3.1 Eq. (1) and §6.3 Table 2).  The sliding-window threshold is read as
 * the mean of the last w token entropies including H, across step boundaries
 * (the pages name the policy without writing it out). */
enum {
  RESET_THRESHOLD_RESET = 0,   /* tau = tau0 if H_step <= H_bar else H_step (SAT over HSE) */
  RESET_THRESHOLD_FIXED = 1,   /* tau = tau0 at every position (Eq. (1))                   */
  RESET_THRESHOLD_WINDOW = 2   /* tau = mean of the last w entropies, including H          */
};

/* A zero-initialised tail (threshold 0, top_p 0) gives ReSET without top-p. */
typedef struct reset_params {
  float tau0;    /* global entropy threshold (nats), used in confident steps        */
  float t_low;   /* temperature below the threshold, > 0                            */
  float t_high;  /* temperature at or above the threshold, > 0                      */
  int w;         /* HSE window: positions 0..w-1 of a step use the last-w mean, 1..256 */
  int threshold; /* RESET_THRESHOLD_*                                                */
  float top_p;   /* nucleus mass in (0, 1); 0 or 1: no truncation                   */
} reset_params;

/* Bytes of the per-row sampler state for M rows and window w. */
size_t reset_state_bytes(int M, int w);

/* Puts every row of `state` at sequence position 0 (asynchronous). */
nvfp4_status reset_state_init(void* state, int M, int w, cudaStream_t stream);

/* Scratch needed by reset_sample for M rows of V logits. */
size_t reset_workspace_bytes(int M, int V);

/*
 * One decode position of the ReSET sampler for M rows (ReSET reading note
 * §4.1 SAT, §4.2 HSE, §4.3; project page "Step-aware temperature scaling"):
 *   H      = entropy (nats, temperature 1) of softmax(logits[r, :]);
 *   a new step starts at this position when step_start[r] != 0 (the previous
 *   token was the step delimiter) and always at the row's first position;
 *   H_step = mean of the last w entropies (including H) while the in-step
 *            position j < w, else the mean of the step's entropies so far;
 *   H_bar  = mean of all entropies of the row so far (including H);
 *   tau    = tau0 if H_step <= H_bar else H_step   (p->threshold RESET_THRESHOLD_RESET;
 *            tau0 for _FIXED, the mean of the last w entropies for _WINDOW);
 *   T      = t_low if H < tau else t_high;
 *   token  = min{ i : sum_{k<=i} exp((l_k - max l)/T) > u[r] * sum_k exp((l_k - max l)/T) }.
 * With 0 < p->top_p < 1 (reading note §6.1: the evaluation samples with
 * top-p 0.95), the sums run over the nucleus only: token i stays iff the sum
 * of exp((l_k - max l)/T) over the logits l_k > l_i is below top_p times the
 * full sum -- the smallest set of most probable tokens that reaches top_p,
 * with every logit tied to its least probable member.  The top-p path adds
 * four launches and computes in integer masses, exp((l - max l)/T) scaled by
 * 2^(62 - ceil(log2 V)) and rounded: deterministic, accurate to ~1e-7 of Z.
 *
 *   logits     device, [M, V] FP32, 16-byte aligned, finite
 *   M          1..64;  V 1 .. 2^24
 *   step_start device, [M] uint8 (may be NULL: no step boundaries)
 *   u          device, [M] FP32 uniforms in [0, 1)
 *   state      device, reset_state_bytes(M, p->w) bytes from reset_state_init (updated)
 *   p          HOST pointer to the parameters (copied at the call); threshold
 *              one of RESET_THRESHOLD_*, top_p in [0, 1] (else NVFP4_ERR_RANGE)
 *   token      device, [M] int32 (written)
 *   H_out      device, [M] FP32 entropies (written; may be NULL)
 *   T_out      device, [M] FP32 chosen temperatures (written; may be NULL)
 *   workspace  device scratch of reset_workspace_bytes(M, V) bytes, 256-byte aligned,
 *              ZEROED ONCE before its first use (every call leaves it ready for
 *              the next); calls that overlap on the GPU must use different workspaces.
 */
nvfp4_status reset_sample(const float* logits, int M, int V, const uint8_t* step_start,
                          const float* u, void* state, const reset_params* p, int32_t* token,
                          float* H_out, float* T_out, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * reset_sample without a workspace argument: same inputs, outputs and rule as
 * reset_sample.  The ReSET pages have no counterpart to this function; it is
 * for callers that cannot allocate device memory -- for example a plugin
 * inside a serving engine that owns every device allocation through its own
 * pool and only hands out fixed input/output buffers, or a latency-critical
 * decode loop that must not call cudaMalloc because it synchronizes the device.
 *
 * Rows of up to 262,144 logits (one thread-block cluster a row, with or
 * without top-p) need no scratch.  Longer rows take a multi-launch path whose
 * scratch (per-row counters, per-chunk partial sums, the top-p records and
 * histograms) lives in a 1,217,280-byte array that the library reserves
 * statically on every GPU that loads it, until the process exits.  Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library routine.
 *   Limit (V > 262,144 only): M * ceil(V / 2048) <= 4096 (M = 8 allows V up
 *          to 1,048,576); larger calls return NVFP4_ERR_SHAPE without
 *          launching anything.
 *   The first call on a device looks up that device's copy of the array
 *   (cudaGetSymbolAddress); make it before any stream capture on that device.
 *   Every call with V > 262,144 uses the same array and clears its counters
 *   (a 256-byte memset on `stream`); such calls that overlap on the GPU (for
 *   example on two unordered streams) race and give wrong results -- order
 *   them.
 */
nvfp4_status reset_sample_noalloc(const float* logits, int M, int V, const uint8_t* step_start,
                                  const float* u, void* state, const reset_params* p, int32_t* token,
                                  float* H_out, float* T_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
