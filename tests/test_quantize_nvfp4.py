"""bi_quantize_nvfp4 on the GPU: codes and scales against the oracle's exact
quantiser (equal everywhere but within binary32 rounding of a rounding
boundary), row-local (batch-invariant), and feeding bi_gemm_nvfp4 end to end.

The quantiser is the activation side of vLLM PR #39912's invariance test
(scaled_fp4_quant with the full tensor's global scale, reused for row slices).
"""
import os

import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, bits_of, check_quant_against_oracle, to_dev, to_dev_bf16, \
    unswizzle_block_scales

pytestmark = pytest.mark.gpu


def gpu_quant(bi, Xbits, gs):
    import torch
    Q, S = bi.quantize_nvfp4(to_dev_bf16(Xbits), gs)
    torch.cuda.synchronize()
    return Q.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (256, 4096), (130, 320), (4096, 4096)])
def test_codes_against_oracle(bi, M, K):
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_FP4_A, M, K)))
    if M > 8:
        x[7] *= 50.0          # outlier row
        x[3, 32:48] = 0.0     # a zero block
    Xb = syn.to_bf16_bits(x)
    gs = syn.nvfp4_global_scale(syn.bf16_bits_to_f32(Xb))
    Q, S_il = gpu_quant(bi, Xb, gs)
    S = unswizzle_block_scales(S_il, M, K // 16)
    # the binding zero-fills the scale buffer: the padding rows and columns of
    # the interleaved layout stay zero, as the generator pads them
    assert np.array_equal(S_il, syn.swizzle_block_scales(S)), "scale padding"
    # codes within binary32 rounding of a boundary may take the neighbouring
    # code; on N(0,1) data such elements are rare (about one in 10^6)
    check_quant_against_oracle(Xb, gs, Q, S, max_count=max(4, M * K // 100000))


def test_special_values_and_ties(bi):
    """Golden blocks from tests/golden (hand-worked) and tie/saturation values.
    In block F three scaled values lie within 2^-24 of a tie, so the kernel's
    binary32 quotient may land on the tie and take the even neighbour."""
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
        check_quant_against_oracle(Xb, gs, Q, unswizzle_block_scales(S_il, 1, 4))


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
