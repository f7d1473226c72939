"""The C ABI library loads and exports every function include/nvfp4.h declares;
argument errors come back synchronously (no GPU needed for any of this)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_w4a4_decode_gemv_gb300 import build
    from nvfp4_w4a4_decode_gemv_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("nvfp4_quantize_act", "nvfp4_gemv_smallm", "reset_sample", "reset_state_bytes",
                     "reset_state_init", "nvfp4_gemv_workspace_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from nvfp4_w4a4_decode_gemv_gb300 import _lib
    names = _declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} declared in nvfp4.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_status_strings_and_version(lib):
    assert lib.nvfp4_version() >> 16 == 1
    for s in range(7):
        assert lib.nvfp4_status_str(s)


FAKE = 1 << 20       # a 256-byte aligned non-NULL address; never dereferenced: validation fails first


def test_quantize_argument_errors(lib):
    assert lib.nvfp4_quantize_act(FAKE, 2, 24, FAKE, FAKE, FAKE, None) == 2       # K % 16
    assert lib.nvfp4_quantize_act(FAKE, -1, 32, FAKE, FAKE, FAKE, None) == 2
    assert lib.nvfp4_quantize_act(None, 2, 32, FAKE, FAKE, FAKE, None) == 1
    assert lib.nvfp4_quantize_act(FAKE + 8, 2, 32, FAKE, FAKE, FAKE, None) == 3   # x not 16-B aligned
    assert lib.nvfp4_quantize_f32(FAKE, 2, 32, 30, FAKE, FAKE, FAKE, None) == 2   # ld < K


def test_gemv_argument_errors(lib):
    args = lambda M, N, K, x=FAKE, ws=FAKE: (x, FAKE, FAKE, M, FAKE, FAKE, FAKE, N, K, FAKE, ws, 1 << 30, None)
    assert lib.nvfp4_gemv_smallm(*args(9, 256, 256)) == 4            # M > 8
    assert lib.nvfp4_gemv_smallm(*args(0, 256, 256)) == 4
    assert lib.nvfp4_gemv_smallm(*args(1, 256, 272)) == 2            # K % 256
    assert lib.nvfp4_gemv_smallm(*args(1, 0, 256)) == 2
    assert lib.nvfp4_gemv_smallm(*args(1, 256, 256, x=None)) == 1
    assert lib.nvfp4_gemv_smallm(*args(1, 256, 256, x=FAKE + 4)) == 3
    assert lib.nvfp4_gemv_smallm(*args(1, 256, 256, ws=FAKE + 16)) == 3
    for fn in (lib.nvfp4_gemv_smallm, lib.nvfp4_gemv_smallm_cudacore):
        assert fn(*args(9, 256, 256)) == 4
        assert fn(*args(1, 256, 272)) == 2
        assert fn(*args(1, 256, 256, x=None)) == 1
        assert fn(*args(1, 256, 256, ws=FAKE + 16)) == 3
    assert lib.nvfp4_gemv_workspace_bytes(9, 256, 256) == 0
    assert lib.nvfp4_gemv_workspace_bytes(1, 256, 100) == 0


def test_gemm_argument_errors(lib):
    args = lambda M, N, K, x=FAKE, ws=FAKE: (x, FAKE, FAKE, M, FAKE, FAKE, N, K, FAKE, ws, 1 << 30, None)
    assert lib.nvfp4_gemm_packed(*args(129, 256, 256)) == 4          # M > 128
    assert lib.nvfp4_gemm_packed(*args(0, 256, 256)) == 4
    assert lib.nvfp4_gemm_packed(*args(64, 256, 272)) == 2           # K % 256
    assert lib.nvfp4_gemm_packed(*args(64, 0, 256)) == 2
    assert lib.nvfp4_gemm_packed(*args(64, 256, 256, x=None)) == 1
    assert lib.nvfp4_gemm_packed(*args(64, 256, 256, x=FAKE + 8)) == 3
    assert lib.nvfp4_gemm_packed(*args(64, 256, 256, ws=FAKE + 16)) == 3
    assert lib.nvfp4_gemm_workspace_bytes(129, 256, 256) == 0
    assert lib.nvfp4_gemm_workspace_bytes(128, 256, 100) == 0


def test_packed_weight_argument_errors(lib):
    assert lib.nvfp4_packed_weight_bytes(1000, 768) == 8 * 3 * 18432      # ceil(1000/128) tiles x 3 chunks
    assert lib.nvfp4_packed_weight_bytes(128, 256) == 18432
    assert lib.nvfp4_packed_weight_bytes(0, 256) == 0
    assert lib.nvfp4_packed_weight_bytes(128, 200) == 0
    assert lib.nvfp4_pack_weights(FAKE, FAKE, 128, 256, FAKE, 18431, None) == 2   # output too small
    assert lib.nvfp4_pack_weights(None, FAKE, 128, 256, FAKE, 18432, None) == 1
    assert lib.nvfp4_pack_weights(FAKE, FAKE, 128, 264, FAKE, 1 << 30, None) == 2
    assert lib.nvfp4_pack_weights(FAKE, FAKE + 8, 128, 256, FAKE, 1 << 30, None) == 3
    args = lambda M, N, K, w=FAKE: (FAKE, FAKE, FAKE, M, w, FAKE, N, K, FAKE, FAKE, 1 << 30, None)
    assert lib.nvfp4_gemv_smallm_packed(*args(9, 256, 256)) == 4
    assert lib.nvfp4_gemv_smallm_packed(*args(1, 256, 300)) == 2
    assert lib.nvfp4_gemv_smallm_packed(*args(1, 256, 256, w=None)) == 1
    assert lib.nvfp4_gemv_smallm_packed(*args(1, 256, 256, w=FAKE + 8)) == 3


def test_quantize_gemv_argument_errors(lib):
    base = lib.nvfp4_gemv_workspace_bytes(8, 5120, 5120)
    need = lib.nvfp4_quantize_gemv_workspace_bytes(8, 5120, 5120)
    assert need >= base + 8 * 5120 // 2 + 8 * 5120 // 16 + 4          # room for the two-launch route
    assert lib.nvfp4_quantize_gemv_workspace_bytes(9, 5120, 5120) == 0
    assert lib.nvfp4_quantize_gemv_workspace_bytes(1, 5120, 5000) == 0
    args = lambda M, N, K, x=FAKE, xg=None, wsb=1 << 30: (x, M, FAKE, FAKE, N, K, FAKE, xg, FAKE, wsb, None)
    assert lib.nvfp4_quantize_gemv_packed(*args(0, 256, 256)) == 4
    assert lib.nvfp4_quantize_gemv_packed(*args(9, 256, 256)) == 4
    assert lib.nvfp4_quantize_gemv_packed(*args(1, 256, 300)) == 2
    assert lib.nvfp4_quantize_gemv_packed(*args(1, 256, 256, x=None)) == 1
    assert lib.nvfp4_quantize_gemv_packed(*args(1, 256, 256, x=FAKE + 8)) == 3
    assert lib.nvfp4_quantize_gemv_packed(*args(1, 256, 256, xg=FAKE + 2)) == 3
    assert lib.nvfp4_quantize_gemv_packed(*args(8, 5120, 5120, wsb=need - 1)) == 2
    assert lib.nvfp4_quantize_gemv_launches(0, 256, 256) == 0
    assert lib.nvfp4_quantize_gemv_launches(1, 256, 300) == 0
    assert lib.nvfp4_quantize_gemv_launches(8, 5120, 5120) == 2          # M above the one-launch limit


def test_reset_argument_errors(lib):
    from nvfp4_w4a4_decode_gemv_gb300._lib import ResetParams
    p = ResetParams(0.6, 0.3, 1.0, 8)
    call = lambda M, V, prm: lib.reset_sample(FAKE, M, V, None, FAKE, FAKE, ctypes.byref(prm), FAKE, None, None,
                                              FAKE, 1 << 30, None)
    assert call(0, 100, p) == 4
    assert call(65, 100, p) == 4
    assert call(8, 0, p) == 2
    assert call(8, 100, ResetParams(0.6, 0.0, 1.0, 8)) == 4           # T_low must be > 0
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 0)) == 4           # w >= 1
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 8, 3, 0.0)) == 4   # unknown threshold policy
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 8, -1, 0.0)) == 4
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 8, 0, 1.5)) == 4   # top_p in [0, 1]
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 8, 0, -0.1)) == 4
    assert call(8, 100, ResetParams(0.6, 0.3, 1.0, 8, 0, float("nan"))) == 4
    noalloc = lambda prm: lib.reset_sample_noalloc(FAKE, 8, 100, None, FAKE, FAKE, ctypes.byref(prm), FAKE, None,
                                                   None, None)
    assert noalloc(ResetParams(0.6, 0.3, 1.0, 8, 2, 2.0)) == 4
    # the top-p scratch: per-row records and 2048-bin histograms, per-chunk kept sums
    assert lib.reset_workspace_bytes(8, 151936) >= 256 + 8 * 75 * 32 + 8 * (64 + 2048 * 8) + 8 * 75 * 8
    assert lib.reset_state_bytes(8, 8) > 0 and lib.reset_state_bytes(8, 0) == 0
    assert lib.reset_workspace_bytes(8, 151936) > 0
    assert lib.nvfp4_bf16_gemv(FAKE, 9, FAKE, 10, 64, FAKE, None) == 4
    assert lib.nvfp4_bf16_gemv(FAKE, 8, FAKE, 10, 8192, FAKE, None) == 2    # M * K > 51200
    assert lib.nvfp4_f32_to_bf16(FAKE, 12, FAKE, None) == 2
    norm = lib.nvfp4_rms_norm_bf16
    assert norm(FAKE, 2, 6, 8, 1e-6, FAKE, None) == 2                  # K % 4
    assert norm(FAKE, 2, 8, 4, 1e-6, FAKE, None) == 2                  # ld < K
    assert norm(FAKE, 2, 8, 8, -1.0, FAKE, None) == 4                  # eps < 0
    assert norm(None, 2, 8, 8, 1e-6, FAKE, None) == 1
    assert norm(FAKE + 8, 2, 8, 8, 1e-6, FAKE, None) == 3


def test_rms_norm_quantize_argument_errors(lib):
    nq = lib.nvfp4_rms_norm_quantize
    assert nq(FAKE, 2, 24, 32, 1e-6, FAKE, FAKE, FAKE, None, None) == 2          # K % 16
    assert nq(FAKE, 2, 8, 8, 1e-6, FAKE, FAKE, FAKE, None, None) == 2            # K < 16
    assert nq(FAKE, 2, 16400, 16400, 1e-6, FAKE, FAKE, FAKE, None, None) == 2    # K / 16 > 1024
    assert nq(FAKE, 2, 32, 16, 1e-6, FAKE, FAKE, FAKE, None, None) == 2          # ld < K
    assert nq(FAKE, 9, 32, 32, 1e-6, FAKE, FAKE, FAKE, None, None) == 4          # rows > 8
    assert nq(FAKE, 2, 32, 32, -1.0, FAKE, FAKE, FAKE, None, None) == 4          # eps < 0
    assert nq(FAKE, 2, 32, 32, 1e-6, FAKE, FAKE, None, None, None) == 1          # global
    assert nq(None, 2, 32, 32, 1e-6, FAKE, FAKE, FAKE, None, None) == 1
    assert nq(FAKE + 8, 2, 32, 32, 1e-6, FAKE, FAKE, FAKE, None, None) == 3      # x alignment
    assert nq(FAKE, 2, 32, 32, 1e-6, FAKE, FAKE, FAKE, FAKE + 8, None) == 3      # r_out alignment


def test_bf16_gemv_tc_argument_errors(lib):
    g = lib.nvfp4_bf16_gemv_tc
    need = lib.nvfp4_bf16_gemv_workspace_bytes(8, 1000, 5120)
    assert need > 0
    assert lib.nvfp4_bf16_gemv_workspace_bytes(8, 1000, 100) == 0            # K % 64
    assert lib.nvfp4_bf16_gemv_workspace_bytes(9, 1000, 128) == 0            # M > 8
    assert need <= lib.nvfp4_gemv_workspace_bytes(8, 1000, 5120)             # a GEMV workspace serves
    assert g(FAKE, 9, FAKE, 10, 64, FAKE, FAKE, need, None) == 4             # M > 8
    assert g(FAKE, 1, FAKE, 10, 96, FAKE, FAKE, need, None) == 2             # K % 64
    assert g(FAKE, 1, FAKE, 0, 64, FAKE, FAKE, need, None) == 2              # N < 1
    assert g(FAKE, 1, FAKE, 10, 64, FAKE, FAKE, 16, None) == 2               # workspace too small
    assert g(None, 1, FAKE, 10, 64, FAKE, FAKE, need, None) == 1
    assert g(FAKE, 1, FAKE, 10, 64, FAKE, None, need, None) == 1
    assert g(FAKE + 8, 1, FAKE, 10, 64, FAKE, FAKE, need, None) == 3         # x alignment
    assert g(FAKE, 1, FAKE, 10, 64, FAKE, FAKE + 16, need, None) == 3        # workspace alignment


def test_reset_params_layout_matches_header(tmp_path):
    """The ctypes mirror of reset_params has the C struct's size, field offsets
    and RESET_THRESHOLD_* values (compiled against include/nvfp4.h by gcc)."""
    import shutil
    import subprocess
    from nvfp4_w4a4_decode_gemv_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = next((d for d in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include"))
                     if os.path.exists(os.path.join(d, "cuda_runtime_api.h"))), None)
    if not cc or not cuda_inc:
        pytest.skip("needs a C compiler and the CUDA headers")
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "nvfp4.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu %zu %zu %zu %d %d %d\\n", sizeof(reset_params),\n'
        "         offsetof(reset_params, tau0), offsetof(reset_params, t_low), offsetof(reset_params, t_high),\n"
        "         offsetof(reset_params, w), offsetof(reset_params, threshold), offsetof(reset_params, top_p),\n"
        "         RESET_THRESHOLD_RESET, RESET_THRESHOLD_FIXED, RESET_THRESHOLD_WINDOW);\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = _lib.ResetParams
    want = [ctypes.sizeof(P)] + [getattr(P, f).offset for f in ("tau0", "t_low", "t_high", "w", "threshold", "top_p")]
    want += [_lib.THRESHOLD_RESET, _lib.THRESHOLD_FIXED, _lib.THRESHOLD_WINDOW]
    assert got == want
