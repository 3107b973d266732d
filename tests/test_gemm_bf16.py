"""bi_gemm_bf16 on the GPU: parity with the fp64 oracle and bit-exact batch invariance.

Invariance checks follow the vLLM batch-invariance pages: row i of a full-M
call equals the M=1 call on that row (vLLM PR #39912,
test_nvfp4_gemm_batch_invariance); identical repeated runs give one distinct
output (vLLM PR #51292, Test Plan: 8 runs, count distinct outputs); plus row
order and padding rows, which the definition of batch invariance covers
(vllm-ascend guide: independent of batch size and request order).
"""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, bits_of, f64_of, sample_rows, to_dev_bf16

pytestmark = pytest.mark.gpu
RTOL = 1e-2   # |gpu - ref| <= 1e-2 * (|ref| + 1): bf16 output of an fp32 sum


def run(bi, X, W):
    return bi.gemm_bf16(to_dev_bf16(X), to_dev_bf16(W))


def test_exact_on_integer_inputs(bi):
    """Integer inputs in [-8, 8]: every partial sum is an integer below 2^24, so
    the fp32 accumulation is exact whatever its order, and the stored output
    must be exactly the bf16 rounding of the oracle's exact sum."""
    for M, N, K in [(1, 512, 256), (64, 512, 256), (130, 264, 72), (257, 16, 8), (200, 384, 1024)]:
        X = syn.integer_bf16(11, 0, (M, K))
        W = syn.integer_bf16(11, 1, (N, K))
        ref = oracle.gemm_bf16(X, W)
        assert np.abs(ref).max() * 1 < 2 ** 24 and 64 * K < 2 ** 24
        got = bits_of(run(bi, X, W))
        assert np.array_equal(got, oracle.bf16_round_array(ref)), (M, N, K)


def test_small_config_parity_and_m_sweep(bi):
    """K=256, N=512, M = 1..64: every M within tolerance, and every row of every M
    bit-identical to the M=64 call and to the M=1 call on that row."""
    K, N, MMAX = 256, 512, 64
    X, W = syn.gemm_inputs(MMAX, N, K, seed=0)
    ref = oracle.gemm_bf16(X, W)
    Wd = to_dev_bf16(W)
    Xd = to_dev_bf16(X)
    full = bits_of(bi.gemm_bf16(Xd, Wd))
    assert_close_abs1(syn.bf16_bits_to_f32(full).astype(np.float64), ref, RTOL, "M=64")
    for M in range(1, MMAX + 1):
        y = bits_of(bi.gemm_bf16(Xd[:M], Wd))
        assert np.array_equal(y, full[:M]), f"M={M} differs from the M=64 prefix"
    for i in range(MMAX):
        y = bits_of(bi.gemm_bf16(Xd[i:i + 1], Wd))
        assert np.array_equal(y[0], full[i]), f"row {i} differs between M=64 and M=1"
    assert bi.device_status() == bi.BI_OK


def test_permutation_padding_repeat(bi):
    K, N, M = 256, 512, 64
    X, W = syn.gemm_inputs(M, N, K, seed=1)
    Wd = to_dev_bf16(W)
    base = bits_of(bi.gemm_bf16(to_dev_bf16(X), Wd))
    perm = syn.permutation(1, M)
    yp = bits_of(bi.gemm_bf16(to_dev_bf16(X[perm]), Wd))
    assert np.array_equal(yp, base[perm]), "row order changed a row's bits"
    for pad_to in (128, 200, 256):
        Xp = np.concatenate([X, syn.filler_rows(2, pad_to - M, K)])
        y = bits_of(bi.gemm_bf16(to_dev_bf16(Xp), Wd))
        assert np.array_equal(y[:M], base), f"padding to {pad_to} changed real rows"
    outs = {bits_of(bi.gemm_bf16(to_dev_bf16(X), Wd)).tobytes() for _ in range(8)}
    assert len(outs) == 1, f"{len(outs)} distinct outputs over 8 identical runs"


def test_ragged_and_strided(bi):
    """Ragged M, N and K tails; row-strided X and Y views."""
    import torch
    M, N, K = 131, 264, 200
    X, W = syn.gemm_inputs(M, N, K, seed=3)
    ref = oracle.gemm_bf16(X, W)
    Xbig = torch.zeros((M, K + 24), dtype=torch.bfloat16, device="cuda")
    Xbig[:, :K] = to_dev_bf16(X)
    Ybig = torch.full((M, N + 40), 7.0, dtype=torch.bfloat16, device="cuda")
    bi.gemm_bf16(Xbig[:, :K], to_dev_bf16(W), Y=Ybig[:, :N])
    got = f64_of(Ybig[:, :N].contiguous())
    assert_close_abs1(got, ref, RTOL, "ragged/strided")
    assert torch.all(Ybig[:, N:] == 7.0), "wrote past N"
    dense = f64_of(bi.gemm_bf16(to_dev_bf16(X), to_dev_bf16(W)))
    assert np.array_equal(dense, got), "strided call differs from dense call"


def test_k_tail_zero_fill_keeps_row_bits(bi):
    """Rows never see data beyond K: appending columns to X's storage (ld > K) changes nothing."""
    import torch
    M, N, K = 70, 128, 72
    X, W = syn.gemm_inputs(M, N, K, seed=4)
    a = bits_of(bi.gemm_bf16(to_dev_bf16(X), to_dev_bf16(W)))
    Xw = torch.randn((M, K + 56), device="cuda").to(torch.bfloat16) * 100
    Xw[:, :K] = to_dev_bf16(X)
    Ww = torch.randn((N, K + 56), device="cuda").to(torch.bfloat16) * 100
    Ww[:, :K] = to_dev_bf16(W)
    b = bits_of(bi.gemm_bf16(Xw[:, :K], Ww[:, :K]))
    assert np.array_equal(a, b)


SHAPES = {"qkv": (6144, 4096), "gate_up": (24576, 4096), "down": (4096, 12288)}


@pytest.mark.parametrize("layer", list(SHAPES))
def test_qwen3_8b_shapes(bi, layer):
    """Qwen3-8B linear layers at M in {1, 7, 64, 513, 4096, 8192}: sampled rows
    against the oracle; every M's sampled rows bit-equal to M=8192's and to M=1 calls."""
    import torch
    N, K = SHAPES[layer]
    MMAX = 8192
    X, W = syn.gemm_inputs(MMAX, N, K, seed=0)
    Xd, Wd = to_dev_bf16(X), to_dev_bf16(W)
    full = bits_of(bi.gemm_bf16(Xd, Wd))
    rows = sample_rows(MMAX, 14, seed=5)
    ref = oracle.gemm_bf16(X[rows], W)
    assert_close_abs1(syn.bf16_bits_to_f32(full[rows]).astype(np.float64), ref, RTOL, f"{layer} M=8192")
    for M in (1, 7, 64, 513, 4096):
        y = bits_of(bi.gemm_bf16(Xd[:M], Wd))
        assert np.array_equal(y, full[:M]), f"{layer}: M={M} differs from the M=8192 prefix"
    for i in sample_rows(MMAX, 6, seed=6):
        y = bits_of(bi.gemm_bf16(Xd[i:i + 1], Wd))
        assert np.array_equal(y[0], full[i]), f"{layer}: row {i} differs between M=8192 and M=1"
    del Xd, Wd
    torch.cuda.empty_cache()
    assert bi.device_status() == bi.BI_OK


def test_matches_cublas_closely(bi):
    """Sanity check against a different implementation (cuBLAS via torch)."""
    import torch
    X, W = syn.gemm_inputs(300, 1024, 1024, seed=8)
    Xd, Wd = to_dev_bf16(X), to_dev_bf16(W)
    ours = bi.gemm_bf16(Xd, Wd).float()
    theirs = (Xd @ Wd.T).float()
    assert torch.allclose(ours, theirs, rtol=1e-2, atol=1e-2)
