"""ctypes binding of libnvfp4_gb300.so: argument marshalling only.

Every function here forwards device pointers, sizes and the current CUDA
stream to the C ABI declared in include/nvfp4.h and raises if the library
returns an error.  There is no CPU path: if the shared library is missing the
first call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4_gb300.so")

STATUS = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
    4: "NVFP4_ERR_RANGE", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_DEVICE",
}

_c_p = ctypes.c_void_p
_c_i = ctypes.c_int
_c_sz = ctypes.c_size_t


# reset_params.threshold values (RESET_THRESHOLD_* in nvfp4.h)
THRESHOLD_RESET, THRESHOLD_FIXED, THRESHOLD_WINDOW = 0, 1, 2


class ResetParams(ctypes.Structure):
    """reset_params; fields left out default to 0 (ReSET threshold, no top-p)."""
    _fields_ = [("tau0", ctypes.c_float), ("t_low", ctypes.c_float), ("t_high", ctypes.c_float), ("w", ctypes.c_int),
                ("threshold", ctypes.c_int), ("top_p", ctypes.c_float)]


# name -> (restype, argtypes); mirrors include/nvfp4.h
SIGNATURES = {
    "nvfp4_status_str": (ctypes.c_char_p, [_c_i]),
    "nvfp4_last_cuda_error": (ctypes.c_char_p, []),
    "nvfp4_version": (_c_i, []),
    "nvfp4_device_status": (_c_i, [ctypes.POINTER(ctypes.c_uint)]),
    "nvfp4_quantize_act": (_c_i, [_c_p, _c_i, _c_i, _c_p, _c_p, _c_p, _c_p]),
    "nvfp4_quantize_f32": (_c_i, [_c_p, _c_i, _c_i, _c_i, _c_p, _c_p, _c_p, _c_p]),
    "nvfp4_silu_mul_quantize": (_c_i, [_c_p, _c_i, _c_i, _c_p, _c_p, _c_p, _c_p]),
    "nvfp4_gemv_workspace_bytes": (_c_sz, [_c_i, _c_i, _c_i]),
    "nvfp4_gemv_smallm": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_p, _c_p, _c_p, _c_i, _c_i, _c_p, _c_p, _c_sz, _c_p]),
    "nvfp4_gemv_smallm_cudacore": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_p, _c_p, _c_p, _c_i, _c_i, _c_p, _c_p, _c_sz,
                                          _c_p]),
    "nvfp4_test_gemv_fault": (None, [ctypes.c_uint, _c_i]),
    "nvfp4_packed_weight_bytes": (_c_sz, [_c_i, _c_i]),
    "nvfp4_gemm_workspace_bytes": (_c_sz, [_c_i, _c_i, _c_i]),
    "nvfp4_gemm_packed": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_p, _c_p, _c_i, _c_i, _c_p, _c_p, _c_sz, _c_p]),
    "nvfp4_pack_weights": (_c_i, [_c_p, _c_p, _c_i, _c_i, _c_p, _c_sz, _c_p]),
    "nvfp4_gemv_smallm_packed": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_p, _c_p, _c_i, _c_i, _c_p, _c_p, _c_sz, _c_p]),
    "nvfp4_quantize_gemv_workspace_bytes": (_c_sz, [_c_i, _c_i, _c_i]),
    "nvfp4_quantize_gemv_launches": (_c_i, [_c_i, _c_i, _c_i]),
    "nvfp4_quantize_gemv_packed": (_c_i, [_c_p, _c_i, _c_p, _c_p, _c_i, _c_i, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "nvfp4_bf16_gemv": (_c_i, [_c_p, _c_i, _c_p, _c_i, _c_i, _c_p, _c_p]),
    "nvfp4_bf16_gemv_workspace_bytes": (ctypes.c_size_t, [_c_i, _c_i, _c_i]),
    "nvfp4_bf16_gemv_tc": (_c_i, [_c_p, _c_i, _c_p, _c_i, _c_i, _c_p, _c_p, ctypes.c_size_t, _c_p]),
    "nvfp4_rms_norm_bf16": (_c_i, [_c_p, _c_i, _c_i, _c_i, ctypes.c_float, _c_p, _c_p]),
    "nvfp4_rms_norm_quantize": (_c_i, [_c_p, _c_i, _c_i, _c_i, ctypes.c_float, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "nvfp4_f32_to_bf16": (_c_i, [_c_p, _c_sz, _c_p, _c_p]),
    "reset_state_bytes": (_c_sz, [_c_i, _c_i]),
    "reset_state_init": (_c_i, [_c_p, _c_i, _c_i, _c_p]),
    "reset_workspace_bytes": (_c_sz, [_c_i, _c_i]),
    "reset_sample": (_c_i, [_c_p, _c_i, _c_i, _c_p, _c_p, _c_p, ctypes.POINTER(ResetParams), _c_p, _c_p, _c_p,
                            _c_p, _c_sz, _c_p]),
    "reset_sample_noalloc": (_c_i, [_c_p, _c_i, _c_i, _c_p, _c_p, _c_p, ctypes.POINTER(ResetParams), _c_p, _c_p,
                                    _c_p, _c_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m nvfp4_w4a4_decode_gemv_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(status: int, what: str) -> None:
    if status != 0:
        msg = lib().nvfp4_status_str(status).decode()
        extra = lib().nvfp4_last_cuda_error().decode() if status == 5 else ""
        raise RuntimeError(f"{what} failed: {STATUS.get(status, status)} ({msg}) {extra}".strip())


def ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def stream_handle(stream=None) -> int:
    """The cudaStream_t to launch on: `stream`, else the current stream (read
    through torch's raw accessor when it has one: building a Stream object
    costs microseconds per call)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _cur_device is not None:
        return _raw_stream(_cur_device())
    return torch.cuda.current_stream().cuda_stream
