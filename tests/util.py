"""Shared helpers for the GPU tests (tensor conversion and tolerance checks)."""
import numpy as np

import bi_synth as syn


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(arr: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def bits_of(t) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of(t) -> np.ndarray:
    return syn.bf16_bits_to_f32(bits_of(t)).astype(np.float64)


def assert_close_abs1(gpu: np.ndarray, ref: np.ndarray, rtol: float, what: str = ""):
    """Per element |gpu - ref| <= rtol * (|ref| + 1)."""
    err = np.abs(gpu - ref)
    lim = rtol * (np.abs(ref) + 1.0)
    bad = err > lim
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]} ref={ref[tuple(i)]} (max err/lim {float((err / lim).max()):.3f})")


def assert_close_rel(gpu: np.ndarray, ref: np.ndarray, rtol: float, atol: float, what: str = ""):
    """Per element |gpu - ref| <= rtol * |ref| + atol."""
    err = np.abs(gpu - ref)
    lim = rtol * np.abs(ref) + atol
    bad = err > lim
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]} ref={ref[tuple(i)]}")


def sample_rows(M: int, n: int, seed: int = 0) -> np.ndarray:
    """First, last and n seeded rows of an M-row batch (sorted, unique)."""
    if M <= n + 2:
        return np.arange(M)
    rest = syn.rng(seed, 1000 + M).choice(np.arange(1, M - 1), size=n, replace=False)
    return np.unique(np.concatenate([[0, M - 1], rest]))


def unswizzle_block_scales(il: np.ndarray, R: int, C: int) -> np.ndarray:
    """The interleaved 128x4 scale layout bi_gemm_nvfp4 reads -> row-major [R, C]
    (inverse of bi_synth.swizzle_block_scales)."""
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    t = np.asarray(il[:Rp * Cp]).reshape(Rp // 128, Cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(Rp, Cp)[:R, :C]

