"""Seeded synthetic inputs shaped like the ReSET pages' workloads.

This module draws random numbers and describes workload shapes; it holds none
of the method's arithmetic (no quantization, no products, no entropies).  Both
the CUDA path and the CPU oracle are fed from here.

Shapes: the decode projections of Qwen3-8B and Qwen3-32B (ReSET project page,
table "Kernel-level decode latency (us) for M=1 GEMV"), with gate and up fused
into one gate_up projection of twice the intermediate size.
"""
import numpy as np
import torch

QWEN3_8B = [("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 24576), ("down", 12288, 4096)]
QWEN3_32B = [("qkv", 5120, 10240), ("o", 8192, 5120), ("gate_up", 5120, 51200), ("down", 25600, 5120)]
QWEN3_14B = [("qkv", 5120, 7168), ("o", 5120, 5120), ("gate_up", 5120, 34816), ("down", 17408, 5120)]
LM_HEAD_VOCAB = 151936

W_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_SCALE = 20.0
OUTLIER_SEED = 2


def gemv_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic HBM bytes of one NVFP4 GEMV call: weight codes + scales,
    activation codes + scales, the two global scales and the FP32 output."""
    return N * K // 2 + N * K // 16 + M * K // 2 + M * K // 16 + 8 + 4 * M * N


def quantize_gemv_bytes(M: int, N: int, K: int) -> int:
    """Algorithmic HBM bytes of one quantize-and-multiply call: weight codes +
    scales, the BF16 activation, the weight's global scale and the FP32 output
    (the quantized activation need not leave the chip)."""
    return N * K // 2 + N * K // 16 + 2 * M * K + 4 + 4 * M * N


def quantize_bytes(M: int, K: int) -> int:
    """Algorithmic bytes of one activation quantization: BF16 in, NVFP4 out."""
    return M * K * 2 + M * K // 2 + M * K // 16 + 4


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std) drawn in FP32 from a seeded torch generator, rounded to BF16 (RNE)."""
    x = torch.randn(shape, generator=_gen(seed, device), dtype=torch.float32, device=device)
    return (x * std).to(torch.bfloat16)


def outlier_channels(K: int, seed: int = OUTLIER_SEED) -> torch.Tensor:
    """The ceil(1% * K) channel indices scaled as outliers (seeded permutation)."""
    n = int(np.ceil(OUTLIER_FRACTION * K))
    return torch.randperm(K, generator=_gen(seed))[:n]


def activations(M: int, K: int, seed: int, outliers: bool = True, device="cpu") -> torch.Tensor:
    """X ~ N(0, 1) [M, K]; 1% of the K channels (fixed across rows) scaled x20 in FP32; BF16."""
    x = torch.randn((M, K), generator=_gen(seed, device), dtype=torch.float32, device=device)
    if outliers:
        x[:, outlier_channels(K).to(device)] *= OUTLIER_SCALE
    return x.to(torch.bfloat16)


def weights(N: int, K: int, seed: int, std: float = W_STD, device="cpu") -> torch.Tensor:
    """W ~ N(0, std) [N, K] in BF16."""
    return normal_bf16((N, K), std, seed, device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---- ReSET sampler workload ---------------------------------------------------
SIGMAS = (1.0, 3.0, 8.0)


def reset_sigmas(steps: int, seed: int = 3) -> np.ndarray:
    """Per-step logit scale drawn uniformly from {1, 3, 8}, shared by all rows."""
    rng = np.random.default_rng(seed)
    return np.array(SIGMAS)[rng.integers(0, len(SIGMAS), steps)]


def reset_logits(step: int, M: int, V: int, sigma: float, base_seed: int = 4, device="cpu") -> torch.Tensor:
    """FP32 logits [M, V] ~ N(0, sigma) for one decode step (generator seed base_seed + step)."""
    x = torch.randn((M, V), generator=_gen(base_seed + step, device), dtype=torch.float32, device=device)
    return x * sigma


def reset_boundaries(steps: int, M: int, p: float = 1 / 30, seed: int = 5) -> np.ndarray:
    """uint8 [steps, M]: 1 where a new reasoning step starts; per row the gaps
    between starts are Geometric(p)."""
    rng = np.random.default_rng(seed)
    out = np.zeros((steps, M), dtype=np.uint8)
    for r in range(M):
        t = int(rng.geometric(p))
        while t < steps:
            out[t, r] = 1
            t += int(rng.geometric(p))
    return out


def reset_uniforms(steps: int, M: int, seed: int = 6) -> np.ndarray:
    """u in [0, 1), float32 [steps, M], from a PCG64 stream."""
    return np.random.Generator(np.random.PCG64(seed)).random((steps, M), dtype=np.float64).astype(np.float32)


# ---- full decode step ---------------------------------------------------------
def decode_weight_std(K: int, proj: str) -> float:
    """Weight scale for the chained decode step: 1/sqrt(K) keeps every layer's
    output O(1) (1.3/sqrt(K) for gate_up, so that SiLU(gate)*up keeps unit
    scale); NVFP4 is scale-invariant per tensor, so this changes no kernel's work."""
    return (1.3 if proj == "gate_up" else 1.0) / float(np.sqrt(K))
