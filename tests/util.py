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


# The quantiser kernel evaluates amax*gs/6 and x*gs/value(s) in binary32 with
# two roundings each (amax/6 then *gs; gs/value(s) then x*), so its quotient is
# within 2^-23 of the exact one, relatively. A code (or scale) can therefore
# differ from the exact definition's only where the exact value lies that close
# to the midpoint between the two codes; the margin below is twice that.
QUANT_BOUNDARY_REL = 2.0 ** -22


def check_quant_against_oracle(Xb: np.ndarray, gs, Q: np.ndarray, S: np.ndarray, max_count=None):
    """Compare a quantiser's packed codes Q [M, K/2] and row-major scales S
    [M, K/16] with the oracle (the exact definition). Every code and scale must
    match, except where the exact scaled value is within QUANT_BOUNDARY_REL of
    the midpoint between the two codes, where the neighbouring code is also
    accepted. A block whose scale is such a neighbour has its codes checked
    against the oracle's codes for that scale. Returns (scales_off, codes_off);
    asserts codes_off + scales_off <= max_count when given."""
    import oracle
    M, K = Xb.shape
    Qo, So = oracle.quantize_nvfp4(Xb, gs)
    g = float(np.float32(gs))
    x = syn.bf16_bits_to_f32(Xb).astype(np.float64)
    e4 = syn._E4M3
    sd = np.argwhere(S != So)
    for i, b in sd:
        a, o = int(S[i, b]), int(So[i, b])
        assert a < 0x7F and o < 0x7F and abs(a - o) == 1, f"scale ({i},{b}): {a:#x} vs {o:#x}"
        v = np.max(np.abs(x[i, 16 * b:16 * b + 16])) * g / 6.0
        mid = (e4[a] + e4[o]) / 2
        assert abs(v - mid) <= QUANT_BOUNDARY_REL * mid, f"scale ({i},{b}): {a:#x} vs {o:#x}, value {v}"
    Qr = oracle.quantize_nvfp4_codes(Xb, gs, S) if len(sd) else Qo
    unpack = lambda q: np.stack([q & 15, q >> 4], axis=-1).reshape(M, K).astype(np.int64)
    ck, cr = unpack(Q), unpack(Qr)
    e2 = syn._E2M1
    mag = lambda c: e2[c & 7]
    cd = np.argwhere(ck != cr)
    for i, k in cd:
        a, o = int(ck[i, k]), int(cr[i, k])
        assert abs(int(a & 7) - int(o & 7)) == 1 and ((a ^ o) & 8 == 0 or (a & 7) == 0 or (o & 7) == 0), \
            f"code ({i},{k}): {a} vs {o}"
        sv = e4[int(S[i, k // 16])]
        y = abs(x[i, k] * g / sv)
        mid = (mag(a) + mag(o)) / 2
        assert abs(y - mid) <= QUANT_BOUNDARY_REL * mid, f"code ({i},{k}): {a} vs {o}, scaled value {y}"
    if max_count is not None:
        assert len(sd) + len(cd) <= max_count, f"{len(sd)} scales and {len(cd)} codes at a boundary"
    return len(sd), len(cd)
