"""fp64 CPU oracle for the batch-invariant linear layer and RMSNorm.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are its only callers. The product library never
imports, links or runs anything here, and this package imports nothing from
the product (the seeded input generator ``bi_synth`` is the one module both
sides use).

The arithmetic lives in ``oracle.c`` (plain loops, fp64, one sequential sum per
output element). This module compiles it with the host C compiler and wraps it
with numpy arrays.

Parity pins (see tests/test_oracle.py): every routine here is checked against
brute force in exact rational arithmetic on small integer / dyadic inputs,
closed forms and the format definitions; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _liboracle.so (OpenMP if the compiler has it).

    -ffp-contract=off keeps every multiply and add separately rounded (no FMA
    contraction), so results are identical on x86-64 and aarch64 hosts."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
            lib.oracle_gemm_bf16.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64]
            lib.oracle_grouped_gemm_bf16.argtypes = [ctypes.c_int32, P, I64, I64, P, P, P]
            lib.oracle_gemm_nvfp4.argtypes = [I64, I64, I64, P, P, P, P, D, P]
            lib.oracle_rmsnorm.argtypes = [I64, I64, P, P, P, D, P, P]
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint]
            lib.oracle_e2m1_value.restype = D
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint]
            lib.oracle_e4m3_value.restype = D
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_value.restype = D
            lib.oracle_bf16_round.argtypes = [D]
            lib.oracle_bf16_round.restype = ctypes.c_uint16
            lib.oracle_bf16_round_array.argtypes = [I64, P, P]
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_quantize_nvfp4.argtypes = [I64, I64, P, ctypes.c_float, P, P]
            lib.oracle_quantize_nvfp4_codes.argtypes = [I64, I64, P, ctypes.c_float, P, P]
            lib.oracle_moe_topk_softmax.argtypes = [I64, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int, P, P]
            lib.oracle_moe_align.argtypes = [I64, ctypes.c_int32, ctypes.c_int32, P, P, P, P]
            lib.oracle_silu_mul.argtypes = [I64, I64, P, P]
            lib.oracle_moe_combine.argtypes = [I64, ctypes.c_int32, I64, P, P, P, P]
            lib.oracle_rank_sum_rmsnorm.argtypes = [ctypes.c_int32, I64, I64, P, P, P, D, P, P, P]
            lib.oracle_attention_decode.argtypes = [I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, D, P]
            lib.oracle_attention_extend.argtypes = [I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, D, P]
            lib.oracle_e4m3_encode.argtypes = [D]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint
            lib.oracle_e2m1_encode.argtypes = [D]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint
            lib.oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    """OpenMP threads the oracle's loops use."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    """Use n OpenMP threads from now on (timing only: each output element is
    one sequential sum, so results do not depend on the thread count)."""
    _load().oracle_set_threads(int(n))


def gemm_bf16(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Y = X W^T in fp64 from bf16 bit patterns X [M,K], W [N,K]."""
    X, W = _c(X, np.uint16), _c(W, np.uint16)
    M, K = X.shape
    N, K2 = W.shape
    assert K == K2
    Y = np.zeros((M, N), dtype=np.float64)
    if M and N:
        _load().oracle_gemm_bf16(M, N, K, _p(X), K, _p(W), K, _p(Y), N)
    return Y


def grouped_gemm_bf16(X: np.ndarray, W: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Per-expert Y[r] = X[r] W[e]^T for rows r in [offsets[e], offsets[e+1])."""
    X, W, off = _c(X, np.uint16), _c(W, np.uint16), _c(offsets, np.int32)
    E, N, K = W.shape
    rows = int(off[-1])
    assert X.shape == (rows, K) and len(off) == E + 1
    Y = np.zeros((rows, N), dtype=np.float64)
    if rows and N:
        _load().oracle_grouped_gemm_bf16(E, _p(off), N, K, _p(X), _p(W), _p(Y))
    return Y


def gemm_nvfp4(A, SA, B, SB, alpha) -> np.ndarray:
    """Y = alpha * dequant(A) dequant(B)^T in fp64; scales row-major [rows, K/16]."""
    A, SA, B, SB = (_c(t, np.uint8) for t in (A, SA, B, SB))
    M, KB = A.shape
    N = B.shape[0]
    K = KB * 2
    assert B.shape == (N, KB) and SA.shape == (M, K // 16) and SB.shape == (N, K // 16)
    Y = np.zeros((M, N), dtype=np.float64)
    if M and N:
        _load().oracle_gemm_nvfp4(M, N, K, _p(A), _p(SA), _p(B), _p(SB), float(alpha), _p(Y))
    return Y


def rmsnorm(x, w, eps: float, residual=None):
    """RMSNorm of bf16 rows (optionally after the residual add).

    Returns (y fp64 [M,H], h_bits uint16 [M,H] or None), where h_bits is the
    rounded sum bf16(x + residual) that the kernel writes back to residual."""
    x, w = _c(x, np.uint16), _c(w, np.uint16)
    M, H = x.shape
    y = np.zeros((M, H), dtype=np.float64)
    h = None
    rp = None
    if residual is not None:
        residual = _c(residual, np.uint16)
        h = np.zeros((M, H), dtype=np.uint16)
        rp = _p(residual)
    if M:
        _load().oracle_rmsnorm(M, H, _p(x), rp, _p(w), float(eps), _p(y),
                               _p(h) if h is not None else None)
    return y, h


def quantize_nvfp4(X: np.ndarray, gs: float):
    """NVFP4 quantisation of bf16 rows X [M,K] with global scale gs: the codes
    and scales of the exact values amax*gs/6 and x*gs/value(s).

    Returns (packed e2m1 codes u8 [M, K/2], e4m3 block scales u8 [M, K/16] row-major)."""
    X = _c(X, np.uint16)
    M, K = X.shape
    assert K % 16 == 0
    Q = np.zeros((M, K // 2), dtype=np.uint8)
    S = np.zeros((M, K // 16), dtype=np.uint8)
    if M:
        _load().oracle_quantize_nvfp4(M, K, _p(X), float(np.float32(gs)), _p(Q), _p(S))
    return Q, S


def quantize_nvfp4_codes(X: np.ndarray, gs: float, S: np.ndarray) -> np.ndarray:
    """The packed e2m1 codes of X [M,K] for given e4m3 block scales S [M, K/16]
    (row-major), by the same definition as quantize_nvfp4."""
    X = _c(X, np.uint16)
    M, K = X.shape
    S = _c(S, np.uint8)
    assert S.shape == (M, K // 16)
    Q = np.zeros((M, K // 2), dtype=np.uint8)
    if M:
        _load().oracle_quantize_nvfp4_codes(M, K, _p(X), float(np.float32(gs)), _p(S), _p(Q))
    return Q


def moe_topk_softmax(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k experts per token (ties to the lower index) and their softmax
    weights (fp64), optionally renormalised over the k chosen."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    assert 1 <= k <= E <= 4096
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    if T:
        _load().oracle_moe_topk_softmax(T, E, k, _p(logits), int(bool(renormalize)), _p(ids), _p(w))
    return ids, w


def moe_align(ids: np.ndarray, E: int):
    """Group (token, rank) pairs by expert, stably by token: (offsets [E+1],
    row_token [T*k], pos [T, k])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    off = np.zeros(E + 1, dtype=np.int32)
    row_token = np.zeros(T * k, dtype=np.int32)
    pos = np.zeros((T, k), dtype=np.int32)
    _load().oracle_moe_align(T, k, E, _p(ids), _p(off), _p(row_token), _p(pos))
    return off, row_token, pos


def silu_mul(gu: np.ndarray) -> np.ndarray:
    """act = silu(gate) * up for bf16 rows [gate | up] (fp64)."""
    gu = _c(gu, np.uint16)
    R, I2 = gu.shape
    act = np.zeros((R, I2 // 2), dtype=np.float64)
    if R:
        _load().oracle_silu_mul(R, I2 // 2, _p(gu), _p(act))
    return act


def moe_combine(Y: np.ndarray, pos: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t] = sum_i w[t,i] * Y[pos[t,i]] in rank order (fp64)."""
    Y, pos, w = _c(Y, np.uint16), _c(pos, np.int32), _c(w, np.float64)
    T, k = pos.shape
    H = Y.shape[1]
    out = np.zeros((T, H), dtype=np.float64)
    if T:
        _load().oracle_moe_combine(T, k, H, _p(Y), _p(pos), _p(w), _p(out))
    return out


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(float(v)))


def rank_sum_rmsnorm(parts, w, eps: float, residual=None):
    """All-reduce of R ranks' bf16 partial rows (exact sum, one bf16 rounding),
    then RMSNorm with optional residual add. parts: bf16 bits [R, M, H].
    Returns (y fp64 [M, H], a_bits [M, H] all-reduced rows, h_bits or None)."""
    parts, w = _c(parts, np.uint16), _c(w, np.uint16)
    R, M, H = parts.shape
    y = np.zeros((M, H), dtype=np.float64)
    a = np.zeros((M, H), dtype=np.uint16)
    h = None
    rp = None
    if residual is not None:
        residual = _c(residual, np.uint16)
        h = np.zeros((M, H), dtype=np.uint16)
        rp = _p(residual)
    if M:
        _load().oracle_rank_sum_rmsnorm(R, M, H, _p(parts), rp, _p(w), float(eps), _p(y), _p(a),
                                        _p(h) if h is not None else None)
    return y, a, h


def attention_decode(Q, K, V, table, lens, scale: float):
    """Softmax attention of one query token per sequence over a paged KV cache (fp64).

    Q bf16 [B, Hq, D]; K, V bf16 [blocks, bs, Hkv, D]; table int32 [B, max_blocks];
    lens int32 [B]. Returns O fp64 [B, Hq, D]."""
    Q, K, V = _c(Q, np.uint16), _c(K, np.uint16), _c(V, np.uint16)
    table, lens = _c(table, np.int32), _c(lens, np.int32)
    B, Hq, D = Q.shape
    _, bs, Hkv, D2 = K.shape
    assert D2 == D and V.shape == K.shape and Hq % Hkv == 0 and table.shape[0] == B and np.all(lens >= 1)
    O = np.zeros((B, Hq, D), dtype=np.float64)
    if B:
        _load().oracle_attention_decode(B, Hq, Hkv, D, bs, table.shape[1], _p(Q), _p(K), _p(V), _p(table),
                                        _p(lens), float(scale), _p(O))
    return O


def attention_extend(Q, cu_q, K, V, table, lens, scale: float):
    """Causal attention of each sequence's new query tokens over its paged KV
    cache (fp64). Q bf16 [total_q, Hq, D]; cu_q int32 [B+1]; K, V bf16
    [blocks, bs, Hkv, D]; table int32 [B, max_blocks]; lens int32 [B] (cached
    length, the new tokens included). Token i of sequence b sits at position
    lens[b] - q_len_b + i and sees tokens 0 .. that position. Returns O fp64
    [total_q, Hq, D]."""
    Q, K, V = _c(Q, np.uint16), _c(K, np.uint16), _c(V, np.uint16)
    cu_q, table, lens = _c(cu_q, np.int32), _c(table, np.int32), _c(lens, np.int32)
    T, Hq, D = Q.shape
    _, bs, Hkv, D2 = K.shape
    B = lens.shape[0]
    assert D2 == D and V.shape == K.shape and Hq % Hkv == 0 and table.shape[0] == B
    assert cu_q.shape == (B + 1,) and cu_q[0] == 0 and cu_q[-1] == T
    assert np.all(np.diff(cu_q) >= 0) and np.all(np.diff(cu_q) <= lens)
    O = np.zeros((T, Hq, D), dtype=np.float64)
    if T:
        _load().oracle_attention_extend(B, Hq, Hkv, D, bs, table.shape[1], _p(Q), _p(cu_q), _p(K), _p(V), _p(table),
                                        _p(lens), float(scale), _p(O))
    return O


def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(code))


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(code))


def bf16_value(bits: int) -> float:
    return float(_load().oracle_bf16_value(bits))


def bf16_round(v: float) -> int:
    return int(_load().oracle_bf16_round(float(v)))


def bf16_round_array(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (round to nearest even) of an fp64 array."""
    v = _c(v, np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    if v.size:
        _load().oracle_bf16_round_array(v.size, _p(v), _p(out))
    return out
