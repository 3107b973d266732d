"""bi_gemm_nvfp4 on the GPU: parity with the fp64 oracle (dequantise, then
multiply) and bit-exact batch invariance.

The invariance check is the one in vLLM PR #39912 ("NVFP4 CUTLASS batch
invariant mode", test_nvfp4_gemm_batch_invariance): quantise the full A once
with its global scale, then for each row i compare the full-M output row with
a call on A[i:i+1] quantised with the same global scale.
"""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, bits_of, sample_rows, to_dev

pytestmark = pytest.mark.gpu
RTOL = 3e-2


def run(bi, A, SA, B, SB, alpha):
    """SA, SB row-major [rows, K/16]; converted to the interleaved layout here."""
    return bits_of(bi.gemm_nvfp4(to_dev(A), to_dev(syn.swizzle_block_scales(SA)), to_dev(B),
                                 to_dev(syn.swizzle_block_scales(SB)), float(alpha)))


def test_exact_unit_scales(bi):
    """Unit scales (e4m3 0x38) and alpha 1: products are multiples of 1/4 and
    sums stay far below 2^22, so the fp32 result is exact and the output must
    be bf16(oracle) bit for bit."""
    g = syn.rng(21, 0)
    for M, N, K in [(1, 256, 256), (70, 512, 512), (130, 264, 320)]:
        A = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
        B = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        SA = np.full((M, K // 16), 0x38, dtype=np.uint8)
        SB = np.full((N, K // 16), 0x38, dtype=np.uint8)
        ref = oracle.gemm_nvfp4(A, SA, B, SB, 1.0)
        got = run(bi, A, SA, B, SB, 1.0)
        assert np.array_equal(got, oracle.bf16_round_array(ref)), (M, N, K)


def test_exact_power_of_two_scales(bi):
    """Scales 0.5, 1, 2 and 4 (and alpha a power of two) keep every term a short
    dyadic number: the sum is exact in fp32, so the result is exact. Catches a
    wrong scale layout (row, column or nibble) bit for bit."""
    g = syn.rng(22, 0)
    M, N, K = 200, 384, 1024
    A = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    codes = np.array([0x30, 0x38, 0x40, 0x48], dtype=np.uint8)
    SA = codes[g.integers(0, 4, size=(M, K // 16))]
    SB = codes[g.integers(0, 4, size=(N, K // 16))]
    ref = oracle.gemm_nvfp4(A, SA, B, SB, 0.125)
    got = run(bi, A, SA, B, SB, 0.125)
    assert np.array_equal(got, oracle.bf16_round_array(ref))


def test_single_scale_block_sensitivity(bi):
    """Change one scale of A and one of B: only the matching row / column may change."""
    g = syn.rng(23, 0)
    M, N, K = 130, 264, 512
    A = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    SA = np.full((M, K // 16), 0x38, dtype=np.uint8)
    SB = np.full((N, K // 16), 0x38, dtype=np.uint8)
    base = run(bi, A, SA, B, SB, 1.0)
    SA2 = SA.copy()
    SA2[77, 19] = 0x40
    SB2 = SB.copy()
    SB2[201, 5] = 0x30
    y = run(bi, A, SA2, B, SB2, 1.0)
    ref = oracle.gemm_nvfp4(A, SA2, B, SB2, 1.0)
    assert np.array_equal(y, oracle.bf16_round_array(ref))
    diff = np.argwhere(y != base)
    assert set(diff[:, 0]) <= {77} | set(range(M)) and set(diff[:, 1]) <= {201} | set(range(N))
    assert all(r == 77 or c == 201 for r, c in diff)


@pytest.mark.parametrize("M", [1, 16, 256, 4096])
def test_config_parity(bi, M):
    """K=4096, N=14336: sampled rows against the oracle at every M."""
    N, K = 14336, 4096
    d = syn.nvfp4_inputs(M, N, K, seed=0)
    got = run(bi, d["A"], d["SA"], d["B"], d["SB"], d["alpha"])
    rows = sample_rows(M, 10, seed=M)
    ref = oracle.gemm_nvfp4(d["A"][rows], d["SA"][rows], d["B"], d["SB"], d["alpha"])
    assert_close_abs1(syn.bf16_bits_to_f32(got[rows]).astype(np.float64), ref, RTOL, f"nvfp4 M={M}")


def test_batch_invariance(bi):
    """Row i of the M=4096 call equals the M=1 call on row i (same global
    scale), every M in {1, 16, 256} is a prefix of M=4096, and 8 runs agree."""
    N, K, MMAX = 14336, 4096, 4096
    d = syn.nvfp4_inputs(MMAX, N, K, seed=1)
    Bd, SBd = to_dev(d["B"]), to_dev(d["SB_il"])

    def call(rows):
        return bits_of(bi.gemm_nvfp4(to_dev(d["A"][rows]), to_dev(syn.swizzle_block_scales(d["SA"][rows])),
                                     Bd, SBd, float(d["alpha"])))
    full = call(np.arange(MMAX))
    for M in (1, 16, 256):
        assert np.array_equal(call(np.arange(M)), full[:M]), f"M={M} is not a prefix of M=4096"
    for i in sample_rows(MMAX, 8, seed=2):
        assert np.array_equal(call(np.array([i]))[0], full[i]), f"row {i} differs between M=4096 and M=1"
    perm = syn.permutation(3, 300)
    assert np.array_equal(call(perm), full[perm])
    outs = {call(np.arange(300)).tobytes() for _ in range(8)}
    assert len(outs) == 1
    assert bi.device_status() == bi.BI_OK
