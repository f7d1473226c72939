"""Python face of the C ABI: the same names as include/nvfp4.h, taking torch
CUDA tensors.  Argument marshalling only -- allocation of outputs and
workspaces with torch, then one call into libnvfp4_gb300.so on the current
stream.  Every computation runs in the library's CUDA kernels.
"""
import ctypes
import weakref

import torch

from ._lib import THRESHOLD_FIXED, THRESHOLD_RESET, THRESHOLD_WINDOW, ResetParams, check, lib, ptr, stream_handle

__all__ = [
    "nvfp4_quantize_act", "nvfp4_quantize_f32", "nvfp4_silu_mul_quantize", "nvfp4_gemv_smallm",
    "nvfp4_gemv_smallm_cudacore", "DEVERR_FLAG_TIMEOUT", "nvfp4_gemm_packed", "nvfp4_gemm_workspace_bytes",
    "nvfp4_gemv_workspace_bytes", "nvfp4_packed_weight_bytes", "nvfp4_pack_weights", "nvfp4_gemv_smallm_packed",
    "NVFP4PackedWeight", "nvfp4_quantize_gemv_packed", "nvfp4_quantize_gemv_workspace_bytes",
    "nvfp4_quantize_gemv_launches", "nvfp4_bf16_gemv", "nvfp4_bf16_gemv_tc", "nvfp4_bf16_gemv_workspace_bytes",
    "nvfp4_rms_norm_bf16", "nvfp4_rms_norm_quantize", "nvfp4_f32_to_bf16",
    "reset_state_bytes",
    "reset_state_init", "reset_workspace_bytes", "reset_sample", "reset_sample_noalloc", "device_status", "GemvWorkspace",
    "NVFP4Tensor", "ResetSampler",
]


class NVFP4Tensor:
    """codes uint8 [rows, K/2], scales uint8 [rows, K/16], global float32 [1] (all on the device)."""

    def __init__(self, codes, scales, global_scale):
        self.codes, self.scales, self.global_scale = codes, scales, global_scale

    @classmethod
    def empty(cls, rows: int, K: int, device="cuda"):
        return cls(torch.empty((rows, K // 2), dtype=torch.uint8, device=device),
                   torch.empty((rows, K // 16), dtype=torch.uint8, device=device),
                   torch.empty((1,), dtype=torch.float32, device=device))

    @property
    def rows(self):
        return self.codes.shape[0]

    @property
    def K(self):
        return self.codes.shape[1] * 2


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


def nvfp4_quantize_act(x_bf16: torch.Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    """BF16 [rows, K] -> NVFP4 (codes, scales, global)."""
    _need_cuda(x_bf16)
    if x_bf16.dtype != torch.bfloat16 or x_bf16.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    rows, K = x_bf16.shape
    out = out or NVFP4Tensor.empty(rows, K, x_bf16.device)
    check(lib().nvfp4_quantize_act(ptr(x_bf16), rows, K, ptr(out.codes), ptr(out.scales), ptr(out.global_scale),
                                   stream_handle(stream)), "nvfp4_quantize_act")
    return out


def nvfp4_quantize_f32(x: torch.Tensor, K: int | None = None, out: NVFP4Tensor | None = None,
                       stream=None) -> NVFP4Tensor:
    """FP32 rows (first K columns of a row-major [rows, ld] tensor) -> BF16 (RNE) -> NVFP4."""
    _need_cuda(x)
    if x.dtype != torch.float32 or x.dim() != 2:
        raise ValueError("x must be a 2-D float32 tensor")
    rows, ld = x.shape
    K = ld if K is None else K
    out = out or NVFP4Tensor.empty(rows, K, x.device)
    check(lib().nvfp4_quantize_f32(ptr(x), rows, K, ld, ptr(out.codes), ptr(out.scales), ptr(out.global_scale),
                                   stream_handle(stream)), "nvfp4_quantize_f32")
    return out


def nvfp4_silu_mul_quantize(gate_up: torch.Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    """FP32 [rows, 2I] -> BF16(SiLU(gate) * up) -> NVFP4 [rows, I]."""
    _need_cuda(gate_up)
    rows, two_i = gate_up.shape
    inter = two_i // 2
    out = out or NVFP4Tensor.empty(rows, inter, gate_up.device)
    check(lib().nvfp4_silu_mul_quantize(ptr(gate_up), rows, inter, ptr(out.codes), ptr(out.scales),
                                        ptr(out.global_scale), stream_handle(stream)), "nvfp4_silu_mul_quantize")
    return out


def nvfp4_gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_gemv_workspace_bytes(M, N, K))


# Device error bit of a GEMV CTA whose wait for another CTA's partial sum gave up
# (nvfp4_device_status); the GEMV workspaces must be zeroed again after it.
DEVERR_FLAG_TIMEOUT = 4

_live_workspaces = weakref.WeakSet()


class GemvWorkspace:
    """A zero-initialised GEMV workspace that grows on demand (re-zeroed when it
    grows, and by device_status() after a GEMV wait gave up)."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = torch.zeros(0, dtype=torch.uint8, device=device)
        _live_workspaces.add(self)

    def get(self, M, N, K) -> torch.Tensor:
        need = nvfp4_gemv_workspace_bytes(M, N, K)
        if need == 0:
            raise ValueError(f"unsupported GEMV shape M={M} N={N} K={K}")
        return self.get_bytes(need)

    def get_bytes(self, need: int) -> torch.Tensor:
        if self.buf.numel() < need:
            self.buf = torch.zeros(need + 4096, dtype=torch.uint8, device=self.device)
        return self.buf

    def rezero(self) -> None:
        self.buf.zero_()


_default_ws: dict = {}


def _ws_for(device) -> GemvWorkspace:
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    if key not in _default_ws:
        _default_ws[key] = GemvWorkspace(device)
    return _default_ws[key]


def nvfp4_gemv_smallm(x: NVFP4Tensor, w: NVFP4Tensor, y: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] = dequant(x) @ dequant(w)^T in FP32."""
    M, N, K = x.rows, w.rows, x.K
    if w.K != K:
        raise ValueError("x and w disagree on K")
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.codes.device)
    ws = workspace if workspace is not None else _ws_for(x.codes.device).get(M, N, K)
    check(lib().nvfp4_gemv_smallm(ptr(x.codes), ptr(x.scales), ptr(x.global_scale), M, ptr(w.codes), ptr(w.scales),
                                  ptr(w.global_scale), N, K, ptr(y), ptr(ws), ws.numel(), stream_handle(stream)),
          "nvfp4_gemv_smallm")
    return y


def nvfp4_gemv_smallm_cudacore(x: NVFP4Tensor, w: NVFP4Tensor, y: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """nvfp4_gemv_smallm on the library's second, CUDA-core kernel (a cross-check, not the fast path)."""
    M, N, K = x.rows, w.rows, x.K
    if w.K != K:
        raise ValueError("x and w disagree on K")
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.codes.device)
    ws = workspace if workspace is not None else _ws_for(x.codes.device).get(M, N, K)
    check(lib().nvfp4_gemv_smallm_cudacore(ptr(x.codes), ptr(x.scales), ptr(x.global_scale), M, ptr(w.codes),
                                           ptr(w.scales), ptr(w.global_scale), N, K, ptr(y), ptr(ws), ws.numel(),
                                           stream_handle(stream)), "nvfp4_gemv_smallm_cudacore")
    return y


class NVFP4PackedWeight:
    """An NVFP4 weight [N, K] in the packed layout of nvfp4_pack_weights: packed uint8 [bytes], global float32 [1]."""

    def __init__(self, packed, global_scale, N: int, K: int):
        self.packed, self.global_scale, self.N, self.K = packed, global_scale, N, K


def nvfp4_packed_weight_bytes(N: int, K: int) -> int:
    return int(lib().nvfp4_packed_weight_bytes(N, K))


def nvfp4_pack_weights(w: NVFP4Tensor, out: torch.Tensor | None = None, stream=None) -> NVFP4PackedWeight:
    """Row-major NVFP4 weight -> packed layout (same bytes, tile-chunk blocks of 18432 B)."""
    N, K = w.rows, w.K
    need = nvfp4_packed_weight_bytes(N, K)
    if need == 0:
        raise ValueError(f"unsupported weight shape N={N} K={K}")
    out = out if out is not None else torch.empty(need, dtype=torch.uint8, device=w.codes.device)
    check(lib().nvfp4_pack_weights(ptr(w.codes), ptr(w.scales), N, K, ptr(out), out.numel(), stream_handle(stream)),
          "nvfp4_pack_weights")
    return NVFP4PackedWeight(out, w.global_scale, N, K)


def nvfp4_gemv_smallm_packed(x: NVFP4Tensor, w: NVFP4PackedWeight, y: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """nvfp4_gemv_smallm with the weight packed."""
    M, N, K = x.rows, w.N, x.K
    if w.K != K:
        raise ValueError("x and w disagree on K")
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.codes.device)
    ws = workspace if workspace is not None else _ws_for(x.codes.device).get(M, N, K)
    check(lib().nvfp4_gemv_smallm_packed(ptr(x.codes), ptr(x.scales), ptr(x.global_scale), M, ptr(w.packed),
                                         ptr(w.global_scale), N, K, ptr(y), ptr(ws), ws.numel(),
                                         stream_handle(stream)), "nvfp4_gemv_smallm_packed")
    return y


def nvfp4_quantize_gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_quantize_gemv_workspace_bytes(M, N, K))


def nvfp4_quantize_gemv_launches(M: int, N: int, K: int) -> int:
    """1 or 2: how nvfp4_quantize_gemv_packed runs the shape; 0 invalid shape, -1 no device."""
    return int(lib().nvfp4_quantize_gemv_launches(M, N, K))


def nvfp4_quantize_gemv_packed(x_bf16: torch.Tensor, w: NVFP4PackedWeight, y: torch.Tensor | None = None,
                               xg_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                               stream=None) -> torch.Tensor:
    """nvfp4_quantize_act(x_bf16) then nvfp4_gemv_smallm_packed, as one call (one launch where it fits)."""
    _need_cuda(x_bf16, y, xg_out)
    if x_bf16.dtype != torch.bfloat16 or x_bf16.dim() != 2:
        raise ValueError("x_bf16 must be a 2-D bfloat16 tensor")
    M, K = x_bf16.shape
    N = w.N
    if w.K != K:
        raise ValueError("x and w disagree on K")
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x_bf16.device)
    if workspace is None:
        need = nvfp4_quantize_gemv_workspace_bytes(M, N, K)
        if need == 0:
            raise ValueError(f"unsupported shape M={M} N={N} K={K}")
        workspace = _ws_for(x_bf16.device).get_bytes(need)
    check(lib().nvfp4_quantize_gemv_packed(ptr(x_bf16), M, ptr(w.packed), ptr(w.global_scale), N, K, ptr(y),
                                           ptr(xg_out), ptr(workspace),
                                           workspace.numel(), stream_handle(stream)), "nvfp4_quantize_gemv_packed")
    return y


def nvfp4_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_gemm_workspace_bytes(M, N, K))


_gemm_ws: dict = {}


def nvfp4_gemm_packed(x: NVFP4Tensor, w: NVFP4PackedWeight, y: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] = dequant(x) @ dequant(w)^T for a prefill-sized batch (M <= 128) on packed weights."""
    M, N, K = x.rows, w.N, x.K
    if w.K != K:
        raise ValueError("x and w disagree on K")
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.codes.device)
    if workspace is None:
        dev = x.codes.device
        key = dev.index if dev.index is not None else torch.cuda.current_device()
        need = nvfp4_gemm_workspace_bytes(M, N, K)
        if need == 0:
            raise ValueError(f"unsupported GEMM shape M={M} N={N} K={K}")
        if key not in _gemm_ws or _gemm_ws[key].numel() < need:
            _gemm_ws[key] = torch.zeros(need, dtype=torch.uint8, device=dev)
        workspace = _gemm_ws[key]
    check(lib().nvfp4_gemm_packed(ptr(x.codes), ptr(x.scales), ptr(x.global_scale), M, ptr(w.packed),
                                  ptr(w.global_scale), N, K, ptr(y), ptr(workspace), workspace.numel(),
                                  stream_handle(stream)), "nvfp4_gemm_packed")
    return y


def nvfp4_bf16_gemv(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ w[N, K]^T for BF16 x, w; FP32 result."""
    _need_cuda(x, w)
    M, K = x.shape
    N = w.shape[0]
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    check(lib().nvfp4_bf16_gemv(ptr(x), M, ptr(w), N, K, ptr(y), stream_handle(stream)), "nvfp4_bf16_gemv")
    return y


def nvfp4_bf16_gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_bf16_gemv_workspace_bytes(M, N, K))


def nvfp4_bf16_gemv_tc(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] @ w[N, K]^T for BF16 x, w on the tensor cores; FP32 result.  `workspace`: a zeroed
    uint8 device tensor of at least nvfp4_bf16_gemv_workspace_bytes(M, N, K) bytes (a GEMV workspace serves)."""
    _need_cuda(x, w)
    M, K = x.shape
    N = w.shape[0]
    y = y if y is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:            # the per-device GEMV workspace (its records region is what this call uses)
        workspace = _ws_for(x.device).get(M, N, 256)
    check(lib().nvfp4_bf16_gemv_tc(ptr(x), M, ptr(w), N, K, ptr(y), ptr(workspace), workspace.numel(),
                                   stream_handle(stream)), "nvfp4_bf16_gemv_tc")
    return y


def nvfp4_rms_norm_bf16(x: torch.Tensor, K: int | None = None, eps: float = 1e-6, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """FP32 rows (first K columns of a row-major [rows, ld] tensor) -> BF16 RMS-normalized [rows, K]."""
    _need_cuda(x)
    if x.dtype != torch.float32 or x.dim() != 2:
        raise ValueError("x must be a 2-D float32 tensor")
    rows, ld = x.shape
    K = ld if K is None else K
    out = out if out is not None else torch.empty((rows, K), dtype=torch.bfloat16, device=x.device)
    check(lib().nvfp4_rms_norm_bf16(ptr(x), rows, K, ld, float(eps), ptr(out), stream_handle(stream)),
          "nvfp4_rms_norm_bf16")
    return out


def nvfp4_rms_norm_quantize(x: torch.Tensor, K: int | None = None, eps: float = 1e-6, out: NVFP4Tensor | None = None,
                            r_out: torch.Tensor | None = None, stream=None) -> NVFP4Tensor:
    """FP32 rows (first K columns of a row-major [rows, ld] tensor) -> BF16 RMS-normalized -> NVFP4, one launch;
    the BF16 rows also go to r_out when it is given."""
    _need_cuda(x)
    if x.dtype != torch.float32 or x.dim() != 2:
        raise ValueError("x must be a 2-D float32 tensor")
    rows, ld = x.shape
    K = ld if K is None else K
    if r_out is not None and (r_out.dtype != torch.bfloat16 or tuple(r_out.shape) != (rows, K)
                              or not r_out.is_contiguous()):
        raise ValueError("r_out must be a contiguous [rows, K] bfloat16 tensor")
    out = out or NVFP4Tensor.empty(rows, K, x.device)
    check(lib().nvfp4_rms_norm_quantize(ptr(x), rows, K, ld, float(eps), ptr(out.codes), ptr(out.scales),
                                        ptr(out.global_scale), ptr(r_out), stream_handle(stream)),
          "nvfp4_rms_norm_quantize")
    return out


def nvfp4_f32_to_bf16(x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need_cuda(x)
    y = y if y is not None else torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    check(lib().nvfp4_f32_to_bf16(ptr(x), x.numel(), ptr(y), stream_handle(stream)), "nvfp4_f32_to_bf16")
    return y


def reset_state_bytes(M: int, w: int) -> int:
    return int(lib().reset_state_bytes(M, w))


def reset_workspace_bytes(M: int, V: int) -> int:
    return int(lib().reset_workspace_bytes(M, V))


def reset_state_init(state: torch.Tensor, M: int, w: int, stream=None) -> None:
    check(lib().reset_state_init(ptr(state), M, w, stream_handle(stream)), "reset_state_init")


def reset_sample(logits, step_start, u, state, params: ResetParams, token, H_out, T_out, workspace, stream=None):
    M, V = logits.shape
    check(lib().reset_sample(ptr(logits), M, V, ptr(step_start), ptr(u), ptr(state), ctypes.byref(params),
                             ptr(token), ptr(H_out), ptr(T_out), ptr(workspace), workspace.numel(),
                             stream_handle(stream)), "reset_sample")


def reset_sample_noalloc(logits, step_start, u, state, params: ResetParams, token, H_out, T_out, stream=None):
    """reset_sample with its scratch in the library's static device array (no
    workspace): for callers that may not allocate device memory.  Limit
    M * ceil(V / 2048) <= 4096; calls that overlap on the GPU race."""
    M, V = logits.shape
    check(lib().reset_sample_noalloc(ptr(logits), M, V, ptr(step_start), ptr(u), ptr(state), ctypes.byref(params),
                                     ptr(token), ptr(H_out), ptr(T_out), stream_handle(stream)),
          "reset_sample_noalloc")


class ResetSampler:
    """Owns the per-row state, the workspace and the outputs of reset_sample for M rows x V logits.

    threshold: "reset" (ReSET's step-aware threshold), "fixed" (tau0 at every
    position) or "window" (the mean of the last w entropies); top_p in (0, 1)
    samples from the nucleus only (1 keeps every token)."""

    THRESHOLDS = {"reset": THRESHOLD_RESET, "fixed": THRESHOLD_FIXED, "window": THRESHOLD_WINDOW}

    def __init__(self, M: int, V: int, tau0=0.6, t_low=0.3, t_high=1.0, w=8, device="cuda", threshold="reset",
                 top_p=1.0):
        self.M, self.V = M, V
        self.params = ResetParams(tau0, t_low, t_high, w, self.THRESHOLDS[threshold], top_p)
        self.state = torch.zeros(reset_state_bytes(M, w), dtype=torch.uint8, device=device)
        self.workspace = torch.zeros(reset_workspace_bytes(M, V), dtype=torch.uint8, device=device)
        self.token = torch.zeros(M, dtype=torch.int32, device=device)
        self.H = torch.zeros(M, dtype=torch.float32, device=device)
        self.T = torch.zeros(M, dtype=torch.float32, device=device)
        reset_state_init(self.state, M, w)

    def __call__(self, logits, step_start, u, stream=None):
        reset_sample(logits, step_start, u, self.state, self.params, self.token, self.H, self.T, self.workspace,
                     stream)
        return self.token, self.H, self.T


def device_status() -> int:
    """Reads and clears the library's device error bits (synchronous).  After a
    GEMV wait gave up (DEVERR_FLAG_TIMEOUT), a late partial sum may sit in a
    workspace: every GemvWorkspace of this process is zeroed again; a caller's
    own workspace tensors must be zeroed by the caller."""
    code = ctypes.c_uint(0)
    check(lib().nvfp4_device_status(ctypes.byref(code)), "nvfp4_device_status")
    if code.value & DEVERR_FLAG_TIMEOUT:
        torch.cuda.synchronize()
        for ws in list(_live_workspaces):
            ws.rezero()
        torch.cuda.synchronize()
    return int(code.value)
