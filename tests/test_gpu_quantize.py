"""GPU quantizer vs the oracle: codes, scales and the global scale bit-exact."""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as Q
from oracle import decode as D
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from tests.gpu_util import bf16_from_f32, bits, to_np

pytestmark = pytest.mark.gpu


def _gpu(x_bf16):
    out = api.nvfp4_quantize_act(x_bf16.cuda())
    return to_np(out.codes), to_np(out.scales), to_np(out.global_scale)[0]


def _check(x_bf16):
    c, s, g = _gpu(x_bf16)
    rc, rs, rg = Q.quantize_bf16(bits(x_bf16))
    assert np.float32(g).view(np.uint32) == np.float32(rg).view(np.uint32), (g, rg)
    assert np.array_equal(s, rs), "scales differ"
    assert np.array_equal(c, rc), f"codes differ at {np.argwhere(c != rc)[:5].tolist()}"


@pytest.mark.parametrize("rows,K", [(1, 512), (1, 16), (3, 48), (8, 4096), (5, 5120), (8, 8192), (8, 25600),
                                    (7, 12288), (2, 25600 + 16)])
def test_activations_bit_exact(rows, K):
    _check(synth.activations(rows, K, seed=11 + rows))


def test_weight_sized_tensor_multi_launch_path():
    # > 16384 blocks: amax kernel + grid quantize + finalize
    _check(synth.weights(2048, 4096, seed=21))
    _check(synth.weights(300, 1040, seed=22))          # ragged: 19500 blocks


def test_hand_worked_example():
    x = np.zeros((2, 48), np.float32)
    x[0, 0:16] = 448 * np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, -6])
    x[0, 16:32] = 224 * np.array([6, -6, 3, -3, 1.5, -1.5, .5, -.5, .25, -.25, 2.5, -2.5, 0, -0.0, 4, -4])
    x[0, 32:36] = [6.375, 1.0, -1.25, 0.75]
    x[1, 1] = -0.0
    x[1, 16:19] = [6 * 2.0 ** -10, -6 * 2.0 ** -10, 2.0 ** -10]
    S = 3 * 2.0 ** -9
    x[1, 32:36] = [6 * S, 1 * S, -0.5 * S, 2 * S]
    c, s, g = _gpu(bf16_from_f32(x))
    assert g == 1.0
    assert s.tolist() == [[0x7E, 0x76, 0x38], [0x00, 0x00, 0x03]]
    el = Q.unpack_codes(c)
    assert el[0, 0:16].tolist() == [0, 0, 1, 2, 2, 2, 3, 4, 4, 4, 5, 6, 6, 6, 7, 15]
    assert el[0, 16:32].tolist() == [7, 15, 5, 13, 3, 11, 1, 9, 0, 8, 4, 12, 0, 8, 6, 14]
    assert el[1, 0:16].tolist() == [0, 8] + [0] * 14
    assert el[1, 32:36].tolist() == [7, 2, 9, 4]


def _adversarial(seed):
    """Blocks whose E2M1 inputs sit exactly on tie points, at power-of-two block
    scales from 2^-9 (E4M3 subnormal) to 256, plus zero blocks, -0.0, scale
    ties and underflowing scales.  g = 1 exactly (one block has amax 2688)."""
    rng = np.random.default_rng(seed)
    blocks = [448 * np.array([6.0] + [0.0] * 15)]            # amax 2688 -> g = 1
    for e in range(-9, 9):
        t = 2.0 ** e
        q = rng.integers(-24, 25, 16).astype(np.float64)
        q[0] = 24                                            # bm = 6 t -> block scale t exactly
        blocks.append(t * q / 4)
    blocks.append(np.zeros(16))
    blocks.append(np.array([-0.0] * 16))
    blocks.append(np.array([6 * 2.0 ** -10, -2.0 ** -10] + [0.0] * 14))      # scale tie 0 vs 2^-9 -> 0
    blocks.append(np.array([18 * 2.0 ** -10, -7 * 2.0 ** -10] + [0.0] * 14))  # scale tie 2^-9 vs 2^-8
    blocks.append(np.array([6.375, -6.375, 5.0, 3.5] + [0.25] * 12))          # scale tie 1 vs 1.125
    x = np.concatenate(blocks).astype(np.float32)
    return x.reshape(1, -1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_adversarial_ties_and_subnormals(seed):
    x = _adversarial(seed)
    _check(bf16_from_f32(x))
    _check(bf16_from_f32(x.reshape(-1, 48)))         # the same 24 blocks as 8 rows of 3


def test_zero_and_empty():
    _check(torch.zeros((4, 64), dtype=torch.bfloat16))
    out = api.nvfp4_quantize_act(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"))
    assert to_np(out.global_scale)[0] == 0.0


def test_f32_rows_with_leading_dimension():
    x = torch.randn((6, 1024 + 64), generator=torch.Generator().manual_seed(5)) * 3
    K = 1024
    out = api.nvfp4_quantize_f32(x.cuda(), K=K)
    rc, rs, rg = Q.quantize_bf16(Q.f32_to_bf16_bits(x[:, :K].numpy()))
    assert np.array_equal(to_np(out.codes), rc) and np.array_equal(to_np(out.scales), rs)
    assert to_np(out.global_scale)[0] == rg


def test_silu_mul_quantize_against_oracle():
    """SiLU uses the device expf (not correctly rounded), so an FP32 product can
    land on the other side of a BF16 rounding boundary than the exact value.
    Elements whose exact value lies within 8 FP32 ulps of such a boundary may
    take either BF16 neighbour; every other code must match exactly."""
    M, inter = 4, 2048
    g = torch.Generator().manual_seed(9)
    gu = torch.randn((M, 2 * inter), generator=g) * 2
    out = api.nvfp4_silu_mul_quantize(gu.cuda())
    a = D.silu_mul(gu.numpy().astype(np.float64))                      # exact-ish FP64
    lo = D.to_bf16_bits(a * (1 - 8 * 2.0 ** -24))
    hi = D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24))
    mid = D.to_bf16_bits(a)
    decisive = (lo == hi) & (lo == mid)
    gpu_c = Q.unpack_codes(to_np(out.codes))
    gpu_g = to_np(out.global_scale)[0]
    # the oracle quantizes its own BF16 values; where the amax element is decisive
    # the global scale must match exactly
    rc, rs, rg = Q.quantize_bf16(mid)
    amax_idx = np.unravel_index(np.argmax(np.abs(Q.bf16_bits_to_f32(mid))), mid.shape)
    assert decisive.mean() > 0.99
    if decisive[amax_idx]:
        assert gpu_g == rg
        # blocks whose 16 values are all decisive have the same scale and codes
        blk = decisive.reshape(M, -1, 16).all(axis=2)
        assert np.array_equal(to_np(out.scales)[blk], rs[blk])
        el_ok = np.repeat(blk, 16, axis=1)
        assert np.array_equal(gpu_c[el_ok], Q.unpack_codes(rc)[el_ok])
        assert blk.mean() > 0.9
