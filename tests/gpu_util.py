"""Helpers shared by the GPU parity tests (test code, not product code)."""
import numpy as np
import torch

from nvfp4_w4a4_decode_gemv_gb300 import synth


def to_np(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def bf16_from_f32(x: np.ndarray) -> torch.Tensor:
    """Exactly representable FP32 values -> BF16 torch tensor (CPU)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "test input must be exact in BF16"
    return b


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, rel=1e-3, abs_=1e-6):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = rel * bound + abs_
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} tol={tol[tuple(i)]!r}")


GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape`/`dtype` with GUARD pattern bytes on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.nbytes = n
        self.buf = torch.full((2 * GUARD + n,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self, what):
        b = to_np(self.buf)
        head, tail = b[:GUARD], b[GUARD + self.nbytes:]
        assert (head == PATTERN).all(), f"{what}: {np.count_nonzero(head != PATTERN)} bytes written before the output"
        assert (tail == PATTERN).all(), f"{what}: {np.count_nonzero(tail != PATTERN)} bytes written after the output"
