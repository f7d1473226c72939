"""Glue of one synthetic decode step around the NVFP4 projections, plain (FP64).

The pages run the NVFP4 linears of a Qwen3 decoder inside a serving engine
(ReSET project page, "Core contribution" and "See it decode"; reading note
§5.2 and §6.4).  A synthetic stand-in chains, per layer, the four projections
qkv -> o -> gate_up -> down; each GEMV output is rounded to BF16 and
re-quantized to NVFP4 as the next input:
  * the o projection reads the first 8192 columns of the qkv output (the query
    part; no attention is on the path);
  * between gate_up and down sits SiLU(gate) * up, with gate = the first half
    of the gate_up columns and up = the second half;
  * after the last layer a BF16 lm_head GEMV produces the logits that feed the
    ReSET sampler;
  * the inputs of the qkv and gate_up projections (and of the lm_head) are RMS
    normalized first, as in the Qwen3 decoders the pages run (reading note
    §6.1); without it SiLU(gate)*up squares the magnitude at every layer.

Where the CUDA path rounds an FP32 result to BF16 (a decision that feeds the
next quantizer), the oracle rounds its FP64 result to FP32 first and then to
BF16, i.e. it takes that decision in the kernel's precision.

Test infrastructure only (see the package docstring).
"""
import numpy as np

from .nvfp4 import bf16_bits_to_f32, f32_to_bf16_bits


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a / (1 + exp(-a)) in FP64."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def silu_mul(gate_up: np.ndarray) -> np.ndarray:
    """SiLU(gate) * up over [M, 2I] -> [M, I], FP64."""
    gu = np.asarray(gate_up, dtype=np.float64)
    inter = gu.shape[1] // 2
    return silu(gu[:, :inter]) * gu[:, inter:]


def to_bf16_bits(y: np.ndarray) -> np.ndarray:
    """FP64 -> FP32 -> BF16 bits (round to nearest even at each step)."""
    return f32_to_bf16_bits(np.asarray(y, dtype=np.float64).astype(np.float32))


def bf16_gemv(x_bits: np.ndarray, w_bits: np.ndarray):
    """logits[m, n] = sum_k x[m, k] w[n, k] for BF16 x, w, in FP64; with error scale."""
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    w = bf16_bits_to_f32(w_bits).astype(np.float64)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """x[r, k] / sqrt(mean_k x[r, k]^2 + eps) in FP64 (no gain)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
