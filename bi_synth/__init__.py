"""Seeded synthetic inputs for the batch-invariant linear layer and RMSNorm.

This module is the only code shared by the fp64 oracle side and the CUDA side.
It draws random numbers, rounds them to the storage formats the kernels take
(bf16, packed e2m1 + e4m3 block scales) and lays them out; it holds none of the
arithmetic the kernels compute (no products, sums, norms or dequantisation).

Streams: every tensor comes from its own numpy PCG64 stream keyed by
``(seed, tensor_id)``, so a prefix of rows is identical whatever the total
row count (a property the batch-invariance tests rely on).

Shapes and distributions follow the Qwen3-shaped workloads described on the
vLLM batch-invariance pages (tested models Qwen3-8B and Qwen3-30B-A3B, vllm-ascend
"Batch Invariance" guide, Tested Models) and the NVFP4 test of vLLM PR #39912
("NVFP4 CUTLASS batch invariant mode", test_nvfp4_gemm_batch_invariance).
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- streams ---

TID_X, TID_W, TID_RES, TID_NORM_W, TID_OUTLIER, TID_LOGITS, TID_HIDDEN, \
    TID_DOWN_IN, TID_W1, TID_W2, TID_FP4_A, TID_FP4_B, TID_FILL, TID_PERM = range(14)


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    """Independent PCG64 stream for one tensor."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(entropy=seed, spawn_key=(tensor_id,))))


def normal_rows(seed: int, tensor_id: int, rows: int, cols: int, std: float = 1.0,
                mean: float = 0.0) -> np.ndarray:
    """fp32 [rows, cols] N(mean, std^2), drawn row by row from one stream so
    that the first r rows never depend on ``rows``."""
    g = rng(seed, tensor_id)
    a = g.standard_normal((rows, cols), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return a


# ------------------------------------------------------------ bf16 storage ---

def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def integer_bf16(seed: int, tensor_id: int, shape, lo: int = -8, hi: int = 8) -> np.ndarray:
    """bf16 bit patterns of integers drawn uniformly from [lo, hi] (exactly representable)."""
    v = rng(seed, tensor_id).integers(lo, hi + 1, size=shape).astype(np.float32)
    return to_bf16_bits(v)


# --------------------------------------------------------------- GEMM data ---

def gemm_inputs(M: int, N: int, K: int, seed: int = 0):
    """X ~ N(0,1) [M,K] and W ~ N(0,0.02^2) [N,K], both bf16 bits (nn.Linear layout)."""
    X = to_bf16_bits(normal_rows(seed, TID_X, M, K))
    W = to_bf16_bits(normal_rows(seed, TID_W, N, K, std=0.02))
    return X, W


def filler_rows(seed: int, rows: int, cols: int) -> np.ndarray:
    """Random bf16 filler rows used to pad a batch (values unrelated to the real rows)."""
    return to_bf16_bits(normal_rows(seed, TID_FILL, rows, cols, std=3.0))


def permutation(seed: int, n: int) -> np.ndarray:
    return rng(seed, TID_PERM).permutation(n)


# ------------------------------------------------------------ RMSNorm data ---

def rmsnorm_inputs(M: int, H: int, seed: int = 0, outlier_frac: float = 0.01,
                   outlier_scale: float = 50.0):
    """x ~ N(0,1) [M,H] with round(outlier_frac*M) rows scaled by outlier_scale
    before bf16 rounding; residual ~ N(0,1) [M,H]; weight = 1 + N(0, 0.1^2) [H].
    Returns (x, residual, weight) as bf16 bits and the outlier row indices."""
    x = normal_rows(seed, TID_X, M, H)
    n_out = int(round(outlier_frac * M))
    rows = np.sort(rng(seed, TID_OUTLIER).choice(M, size=n_out, replace=False)) if n_out else \
        np.zeros(0, dtype=np.int64)
    x[rows] *= np.float32(outlier_scale)
    res = normal_rows(seed, TID_RES, M, H)
    w = normal_rows(seed, TID_NORM_W, 1, H, std=0.1, mean=1.0)[0]
    return to_bf16_bits(x), to_bf16_bits(res), to_bf16_bits(w), rows


# ----------------------------------------------------------------- MoE data ---

def moe_routing(T: int, E: int = 128, topk: int = 8, seed: int = 0):
    """Top-k expert choice per token from seeded N(0,1) router logits.

    Softmax is monotonic, so the top-k of the softmax equals the top-k of the
    logits; ties go to the lower expert index. Rows are then grouped by expert,
    stably by token. Returns (row_token [T*topk], row_expert [T*topk],
    offsets [E+1] int32, topk_ids [T, topk])."""
    logits = normal_rows(seed, TID_LOGITS, T, E)
    topk_ids = np.argsort(-logits, axis=1, kind="stable")[:, :topk].astype(np.int32)
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    exp = topk_ids.reshape(-1).astype(np.int64)
    order = np.lexsort((tok, exp))          # by expert, then token
    row_token, row_expert = tok[order], exp[order]
    counts = np.bincount(row_expert, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return row_token, row_expert, offsets, topk_ids


def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(len(counts) + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off


def moe_weights(E: int, N: int, K: int, seed: int = 0, tensor_id: int = TID_W1) -> np.ndarray:
    """Expert weights ~ N(0, 0.02^2) [E, N, K] bf16 bits."""
    return to_bf16_bits(normal_rows(seed, tensor_id, E * N, K, std=0.02)).reshape(E, N, K)


# -------------------------------------------------------------- NVFP4 data ---
# Storage formats (OCP Microscaling spec): e2m1 = 1 sign, 2 exponent (bias 1),
# 1 mantissa bit; e4m3 (FN) = 1 sign, 4 exponent (bias 7), 3 mantissa bits,
# no infinities, 0x7F/0xFF NaN. The encoders below are table searches over the
# values each code stands for; round to nearest, ties to the even code.

def _e2m1_code_values() -> np.ndarray:
    v = np.zeros(8, dtype=np.float64)
    for c in range(8):
        e, m = c >> 1, c & 1
        v[c] = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return v


def _e4m3_code_values() -> np.ndarray:
    v = np.zeros(127, dtype=np.float64)       # positive finite codes 0x00..0x7E
    for c in range(127):
        e, m = c >> 3, c & 7
        v[c] = (2.0 ** -6) * (m / 8.0) if e == 0 else (2.0 ** (e - 7)) * (1.0 + m / 8.0)
    return v


_E2M1 = _e2m1_code_values()
_E4M3 = _e4m3_code_values()


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest table value to each magnitude (ties to the even
    index); magnitudes above the table's top saturate to the top code."""
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.clip(np.searchsorted(table, mag, side="left"), 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    dlo = np.abs(mag - table[lo])
    dhi = np.abs(table[hi] - mag)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= table[-1], len(table) - 1, code)
    return code.astype(np.uint8)


def e4m3_encode_pos(v: np.ndarray) -> np.ndarray:
    """Non-negative fp values -> e4m3 codes (RNE, saturating at 448)."""
    return _nearest_code(v, _E4M3)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """fp values in [-6, 6] -> 4-bit e2m1 codes (RNE; sign in bit 3; zero -> 0).

    Counts the midpoints between neighbouring code values that |v| passes; at
    an exact midpoint it passes only when the upper neighbour's code is even
    (ties to even). Same result as the table search, much faster."""
    v = np.asarray(v)
    mag = np.abs(v).astype(np.float64)
    c = np.zeros(mag.shape, dtype=np.uint8)
    for lo in range(7):
        mid = (_E2M1[lo] + _E2M1[lo + 1]) / 2
        c += (mag >= mid) if (lo + 1) % 2 == 0 else (mag > mid)
    return np.where((v < 0) & (c != 0), c | np.uint8(8), c).astype(np.uint8)


def e2m1_encode_by_search(v: np.ndarray) -> np.ndarray:
    """Reference form of e2m1_encode (table search); kept for the generator's tests."""
    v = np.asarray(v, dtype=np.float64)
    c = _nearest_code(np.abs(v), _E2M1)
    return np.where((v < 0) & (c != 0), c | np.uint8(8), c).astype(np.uint8)


def nvfp4_global_scale(x: np.ndarray) -> np.float32:
    """Per-tensor global scale gs = 448*6 / amax(|x|) (fp32); 1 for an all-zero tensor."""
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(np.float32(448.0 * 6.0) / amax)


def nvfp4_quantize(x: np.ndarray, gs: np.float32):
    """Quantise [R, K] values exact in bf16 (K % 16 == 0) with global scale gs.

    Per 16-element block: s = e4m3(amax_block * gs / 6); q = e2m1(x * gs / s),
    q = 0 where s decodes to 0. The quotients are taken in fp64, where the
    products x*gs are exact and the one division cannot move a value across a
    rounding boundary, so the codes are those of the exact values. Returns
    (packed codes u8 [R, K/2] with the even k in the low nibble, block scales
    u8 [R, K/16] row-major)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    R, K = x.shape
    assert K % 16 == 0
    g = np.float64(np.float32(gs))
    blocks = x.reshape(R, K // 16, 16)
    amax = np.max(np.abs(blocks), axis=2)
    s_code = e4m3_encode_pos(amax * g / 6.0)
    s_val = _E4M3[s_code].astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = blocks * g / s_val[:, :, None]
    scaled = np.where(s_val[:, :, None] == 0, 0.0, scaled)
    scaled = np.clip(scaled, -6.0, 6.0)
    q = e2m1_encode(scaled).reshape(R, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, s_code.astype(np.uint8)


def swizzle_block_scales(sf: np.ndarray) -> np.ndarray:
    """Row-major block scales [R, K/16] -> the interleaved 128x4 layout bi_gemm_nvfp4 reads.

    Rows pad to a multiple of 128 and scale columns to a multiple of 4 (zeros).
    Each 512-byte atom holds 128 rows x 4 consecutive scale columns; scale (r, c)
    sits at byte ((r//128)*(Cp//4) + c//4)*512 + (r%32)*16 + ((r%128)//32)*4 + c%4."""
    R, C = sf.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    pad = np.zeros((Rp, Cp), dtype=np.uint8)
    pad[:R, :C] = sf
    # [rb, r1(4), r0(32), cb, c(4)] -> [rb, cb, r0, r1, c]
    t = pad.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(-1)


def nvfp4_inputs(M: int, N: int, K: int, seed: int = 0):
    """A, B from N(0,1) rounded to bf16, quantised with per-tensor global scales.

    The activation global scale is computed once over all M rows; callers that
    take row slices reuse it (the invariance test in vLLM PR #39912 does the
    same). Returns a dict with packed codes, row-major and interleaved scales,
    the global scales and alpha = 1/(gsA*gsB)."""
    a = bf16_bits_to_f32(to_bf16_bits(normal_rows(seed, TID_FP4_A, M, K)))
    b = bf16_bits_to_f32(to_bf16_bits(normal_rows(seed, TID_FP4_B, N, K)))
    gsa, gsb = nvfp4_global_scale(a), nvfp4_global_scale(b)
    qa, sa = nvfp4_quantize(a, gsa)
    qb, sb = nvfp4_quantize(b, gsb)
    alpha = np.float32(np.float32(1.0) / (gsa * gsb))
    return dict(A=qa, SA=sa, SA_il=swizzle_block_scales(sa), B=qb, SB=sb,
                SB_il=swizzle_block_scales(sb), gsa=gsa, gsb=gsb, alpha=alpha, a_f32=a, b_f32=b)
