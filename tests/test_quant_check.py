"""CPU checks of the quantiser comparison used by the GPU tests: it accepts a
binary32 evaluation of the quantiser (the kernel's order of operations), whose
codes leave the exact definition only at rounding boundaries, and it rejects
plausible mistakes planted in that evaluation."""
import numpy as np
import pytest

import bi_synth as syn
from util import check_quant_against_oracle, unswizzle_block_scales


def quant_f32(x: np.ndarray, gs):
    """Binary32 evaluation: s = e4m3(fl(fl(amax/6)*gs)), q = e2m1(fl(x*fl(gs/s)))."""
    f = np.float32
    R, K = x.shape
    blocks = x.astype(f).reshape(R, K // 16, 16)
    amax = np.max(np.abs(blocks), axis=2)
    s = syn.e4m3_encode_pos((amax / f(6.0)).astype(f) * f(gs))
    sv = syn._E4M3[s].astype(f)
    with np.errstate(divide="ignore"):
        inv = np.where(sv == 0, f(0), f(gs) / sv).astype(f)
    y = np.clip((blocks * inv[:, :, None]).astype(f), -6, 6)
    q = syn.e2m1_encode(y).reshape(R, K)
    return (q[:, 0::2] | (q[:, 1::2] << np.uint8(4))).astype(np.uint8), s.astype(np.uint8)


def inputs(M=64, K=1024):
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(syn.normal_rows(9, syn.TID_FP4_A, M, K)))
    x[5] *= 50.0
    Xb = syn.to_bf16_bits(x)
    return Xb, syn.nvfp4_global_scale(syn.bf16_bits_to_f32(Xb))


def test_accepts_binary32_order():
    Xb, gs = inputs()
    Q, S = quant_f32(syn.bf16_bits_to_f32(Xb), gs)
    check_quant_against_oracle(Xb, gs, Q, S, max_count=4)


def test_accepts_golden_block_f():
    """Block F of the golden cases: the binary32 order lands three elements on
    a tie, where the comparison accepts the even neighbour."""
    vals = [0.004425048828125, 0.01519775390625, -0.004425048828125, 0.007598876953125, 0, 0.00885009765625,
            -0.01519775390625] + [0] * 9
    Xb = syn.to_bf16_bits(np.array([vals * 4], dtype=np.float32))
    gs = np.float32(370.75860595703125)
    Q, S = quant_f32(syn.bf16_bits_to_f32(Xb), gs)
    assert check_quant_against_oracle(Xb, gs, Q, S) == (0, 12)


@pytest.mark.parametrize("mistake", ["nibbles_swapped", "scale_up", "code_up", "sign", "wrong_gs"])
def test_rejects_planted_mistakes(mistake):
    Xb, gs = inputs()
    x = syn.bf16_bits_to_f32(Xb)
    Q, S = quant_f32(x, gs)
    if mistake == "nibbles_swapped":
        Q = ((Q >> 4) | (Q << 4)).astype(np.uint8)
    elif mistake == "scale_up":
        S = S.copy()
        S[3, 7] += 1
    elif mistake == "code_up":
        Q = Q.copy()
        Q[2, 10] = (Q[2, 10] & 0xF0) | min((Q[2, 10] & 7) + 1, 7) | (Q[2, 10] & 8)
        if np.array_equal(Q, quant_f32(x, gs)[0]):
            pytest.skip("code already saturated")
    elif mistake == "sign":
        Q = (Q ^ 0x08).astype(np.uint8)
    elif mistake == "wrong_gs":
        Q, S = quant_f32(x, np.float32(gs * 1.01))
    with pytest.raises(AssertionError):
        check_quant_against_oracle(Xb, gs, Q, S)


def test_unswizzle_inverts_swizzle():
    g = syn.rng(3, 0)
    for R, C in ((1, 4), (130, 20), (256, 256)):
        S = g.integers(0, 0x7F, size=(R, C), dtype=np.uint8)
        assert np.array_equal(unswizzle_block_scales(syn.swizzle_block_scales(S), R, C), S)
