"""bi_quantize_nvfp4 on the GPU: codes and scales bit-exact against the
oracle's quantiser (the exact definition), row-local (batch-invariant), and
feeding bi_gemm_nvfp4 end to end.

The quantiser is the activation side of vLLM PR #39912's invariance test
(scaled_fp4_quant with the full tensor's global scale, reused for row slices).
"""
import os

import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, bits_of, to_dev, to_dev_bf16, unswizzle_block_scales

pytestmark = pytest.mark.gpu


def gpu_quant(bi, Xbits, gs):
    import torch
    Q, S = bi.quantize_nvfp4(to_dev_bf16(Xbits), gs)
    torch.cuda.synchronize()
    return Q.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (256, 4096), (130, 320), (4096, 4096)])
def test_bit_exact_against_oracle(bi, M, K):
    """With the outlier row the global scale is a power of two (16), and about
    1 % of the elements lie within a few binary32 ulps of a rounding midpoint
    (many exactly on it): the kernel's exact side decision is exercised often."""
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_FP4_A, M, K)))
    if M > 8:
        x[7] *= 50.0          # outlier row
        x[3, 32:48] = 0.0     # a zero block
    Xb = syn.to_bf16_bits(x)
    gs = syn.nvfp4_global_scale(syn.bf16_bits_to_f32(Xb))
    Q, S_il = gpu_quant(bi, Xb, gs)
    Qo, So = oracle.quantize_nvfp4(Xb, gs)
    assert np.array_equal(Q, Qo), "codes differ"
    assert np.array_equal(unswizzle_block_scales(S_il, M, K // 16), So), "scales differ"
    # the binding zero-fills the scale buffer and the generator pads with zeros,
    # so the whole interleaved buffer must match, padding rows included
    assert np.array_equal(S_il, syn.swizzle_block_scales(So)), "scale padding"


def test_bit_exact_at_the_bench_size_sampled(bi):
    """The size the bench times (M=16384, K=4096: the multi-row grid, two rows
    per step): codes and scales of sampled rows, bit-exact against the oracle
    quantising those rows alone with the full tensor's global scale (the
    quantiser is row-local)."""
    import torch
    M, K = 16384, 4096
    g = torch.Generator(device="cuda").manual_seed(7)
    X = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    X[5000] *= 50.0                                     # an outlier row sets the global scale
    Xb_all = bits_of(X)
    gs = syn.nvfp4_global_scale(syn.bf16_bits_to_f32(Xb_all))
    Q, S_il = bi.quantize_nvfp4(X, gs)
    torch.cuda.synchronize()
    Q, S_il = Q.cpu().numpy(), S_il.cpu().numpy()
    S = unswizzle_block_scales(S_il, M, K // 16)
    rows = [0, 1, 127, 128, 5000, 8191, 8192, 16383]
    Qo, So = oracle.quantize_nvfp4(Xb_all[rows], gs)
    assert np.array_equal(Q[rows], Qo), "codes differ"
    assert np.array_equal(S[rows], So), "scales differ"
    assert bi.device_status() == bi.BI_OK


def test_special_values_and_ties(bi):
    """Golden blocks from tests/golden (hand-worked): ties, saturation, zero
    and subnormal scales, and block F, whose three scaled values lie within
    2^-24 of a tie (a binary32 evaluation lands on the tie)."""
    rows = []
    gss = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_quant_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                _, gs, xs, _, _ = line.split()
                rows.append([float(v) for v in xs.split(",")])
                gss.append(float(gs))
    for r, gs in zip(rows, gss):
        x = np.array(r * 4, dtype=np.float32)[None]          # K = 64
        Xb = syn.to_bf16_bits(x)
        Q, S_il = gpu_quant(bi, Xb, gs)
        Qo, So = oracle.quantize_nvfp4(Xb, gs)
        assert np.array_equal(Q, Qo) and np.array_equal(unswizzle_block_scales(S_il, 1, 4), So), (gs, r)


def test_row_local(bi):
    """A row quantises to the same bytes alone, in a batch, and after permutation."""
    M, K = 300, 1024
    Xb = syn.to_bf16_bits(syn.normal_rows(1, syn.TID_FP4_A, M, K))
    gs = syn.nvfp4_global_scale(syn.bf16_bits_to_f32(Xb))
    Q, _ = gpu_quant(bi, Xb, gs)
    for i in (0, 1, 127, 128, 299):
        Qi, Si = gpu_quant(bi, Xb[i:i + 1], gs)
        assert np.array_equal(Qi[0], Q[i])
    perm = syn.permutation(2, M)
    Qp, _ = gpu_quant(bi, Xb[perm], gs)
    assert np.array_equal(Qp, Q[perm])


def test_feeds_gemm_end_to_end(bi):
    """GPU-quantised activations through bi_gemm_nvfp4 match the oracle's
    quantise-then-dequantise-then-multiply, and each row equals its M=1 run."""
    M, N, K = 200, 1024, 2048
    a = syn.to_bf16_bits(syn.normal_rows(3, syn.TID_FP4_A, M, K))
    d = syn.nvfp4_inputs(1, N, K, seed=3)
    gsa = syn.nvfp4_global_scale(syn.bf16_bits_to_f32(a))
    alpha = np.float32(1.0) / (gsa * d["gsb"])
    import torch
    Q, S = bi.quantize_nvfp4(to_dev_bf16(a), gsa)
    Bd, SBd = to_dev(d["B"]), to_dev(d["SB_il"])
    Y = bits_of(bi.gemm_nvfp4(Q, S, Bd, SBd, float(alpha)))
    Qo, So = oracle.quantize_nvfp4(a, gsa)
    ref = oracle.gemm_nvfp4(Qo, So, d["B"], d["SB"], float(alpha))
    assert_close_abs1(syn.bf16_bits_to_f32(Y).astype(np.float64), ref, 3e-2, "quantise+gemm")
    for i in (0, 57, 199):
        Qi, Si = bi.quantize_nvfp4(to_dev_bf16(a[i:i + 1]), gsa)
        Yi = bits_of(bi.gemm_nvfp4(Qi, Si, Bd, SBd, float(alpha)))
        assert np.array_equal(Yi[0], Y[i])
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_OK
