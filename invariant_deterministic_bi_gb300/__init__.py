"""Python binding of libbi: batch-invariant linear layers and RMSNorm for GB300.

Argument marshalling only: every function here checks dtypes and devices,
takes data pointers, sizes and the current CUDA stream from torch tensors and
calls the matching ``extern "C"`` entry point of ``libbi.so`` (declared in
``include/bi.h``). All arithmetic runs in the library's sm_103a kernels; there
is no CPU or PyTorch fallback. If the library is missing this module raises.

Names follow the C ABI: ``gemm_bf16``, ``grouped_gemm_bf16``, ``gemm_nvfp4``,
``quantize_nvfp4``, ``rmsnorm``, ``plan``, ``device_status``, ``check_wait_timeout``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# BI_LIBRARY=debug selects the debug build (bounds-checked kernels, same results)
LIB_PATH = os.path.join(_HERE, "libbi_debug.so" if os.environ.get("BI_LIBRARY") == "debug" else "libbi.so")

(BI_OK, BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED, BI_ERR_MISALIGNED, BI_ERR_ARCH, BI_ERR_CUDA, BI_ERR_TIMEOUT,
 BI_ERR_BOUNDS) = range(8)
OP_GEMM_BF16, OP_GROUPED_GEMM_BF16, OP_GEMM_NVFP4, OP_RMSNORM, OP_QUANTIZE_NVFP4, OP_GROUPED_GEMM_SILU_BF16 = range(6)

_lock = threading.Lock()
_lib = None


class BiError(RuntimeError):
    """A libbi call returned a non-OK status."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class Plan(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32),
                ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("mma_m", ctypes.c_int32), ("mma_n", ctypes.c_int32), ("mma_k", ctypes.c_int32),
                ("k_steps", ctypes.c_int32), ("split_k", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64),
                ("grid", ctypes.c_int32), ("reduce_tree", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


def load() -> ctypes.CDLL:
    """Load libbi.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbi.so is not built ({LIB_PATH}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        sig = {
            "bi_gemm_bf16": [P, I64, P, I64, P, I64, I64, I64, I64, P],
            "bi_grouped_gemm_bf16": [P, P, P, P, I32, I64, I64, I64, P],
            "bi_grouped_gemm_silu_bf16": [P, P, P, P, I32, I64, I64, I64, P],
            "bi_gemm_nvfp4": [P, P, P, P, F, P, I64, I64, I64, P],
            "bi_rmsnorm": [P, P, P, P, I64, I64, F, P],
            "bi_quantize_nvfp4": [P, I64, F, P, P, I64, I64, P],
            "bi_moe_topk_softmax": [P, I64, I32, I32, I32, P, P, P],
            "bi_moe_align": [P, I64, I32, I32, P, P, P, P],
            "bi_moe_gather": [P, I64, I64, P, I64, P, P],
            "bi_silu_mul": [P, I64, I64, P, P],
            "bi_moe_combine": [P, I64, P, P, I64, I32, I64, P, P],
            "bi_rank_sum_rmsnorm": [P, I32, P, P, P, P, I64, I64, F, P],
            "bi_attention_decode": [P, P, P, P, I32, I64, P, I64, I32, I32, I32, I32, I32, F, P, I64, P, P],
            "bi_attention_decode_workspace_size": [I64, I32, I32],
            "bi_attention_decode_noalloc": [P, P, P, P, I32, I64, P, I64, I32, I32, I32, I32, I32, F, P, P],
            "bi_debug_build": [],
            "bi_last_bounds_line": [],
            "bi_check_bounds": [I32, I32, P],
            "bi_attention_extend": [P, P, I32, P, P, P, I32, I64, P, I64, I32, I32, I32, I32, I32, I32, F, P, P],
            "bi_plan": [I32, I64, I64, I64, I32, ctypes.POINTER(Plan)],
            "bi_device_status": [P],
            "bi_check_wait_timeout": [ctypes.c_uint32, P],
            "bi_status_string": [ctypes.c_int],
            "bi_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.bi_status_string.restype = ctypes.c_char_p
        lib.bi_attention_decode_workspace_size.restype = ctypes.c_int64
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().bi_status_string(status).decode()


def version() -> int:
    return int(load().bi_version())


def _check(status: int, where: str):
    if status != BI_OK:
        raise BiError(status, where)


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def gemm_bf16(X, W, Y=None, stream=None):
    """Y[M,N] = X[M,K] W[N,K]^T (bf16 in/out, fp32 accumulate), batch-invariant.

    X and W may be row-strided views (unit column stride); Y is allocated if None."""
    import torch
    _dev(X, torch.bfloat16, "X"), _dev(W, torch.bfloat16, "W")
    if X.dim() != 2 or W.dim() != 2 or X.shape[1] != W.shape[1]:
        raise ValueError(f"shape mismatch X{tuple(X.shape)} W{tuple(W.shape)}")
    if X.stride(1) != 1 or W.stride(1) != 1:
        raise ValueError("X and W need unit column stride")
    M, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _dev(Y, torch.bfloat16, "Y")
    if Y.shape != (M, N) or Y.stride(1) != 1:
        raise ValueError("Y must be [M, N] with unit column stride")
    _check(load().bi_gemm_bf16(_ptr(X), X.stride(0), _ptr(W), W.stride(0), _ptr(Y), Y.stride(0), M, N, K,
                               _stream(stream)), "bi_gemm_bf16")
    return Y


def grouped_gemm_bf16(X, W, offsets, Y=None, stream=None):
    """Per-expert Y[r] = X[r] W[e]^T for rows r in [offsets[e], offsets[e+1]).

    X [rows,K], W [E,N,K] bf16 (contiguous); offsets int32 [E+1] on the device."""
    import torch
    _dev(X, torch.bfloat16, "X"), _dev(W, torch.bfloat16, "W"), _dev(offsets, torch.int32, "offsets")
    if not (X.is_contiguous() and W.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("X, W and offsets must be contiguous")
    E, N, K = W.shape
    rows = X.shape[0]
    if X.shape[1] != K or offsets.numel() != E + 1:
        raise ValueError("shape mismatch")
    if Y is None:
        Y = torch.empty((rows, N), dtype=torch.bfloat16, device=X.device)
    _dev(Y, torch.bfloat16, "Y")
    if Y.shape != (rows, N) or not Y.is_contiguous():
        raise ValueError("Y must be contiguous [rows, N]")
    _check(load().bi_grouped_gemm_bf16(_ptr(X), _ptr(W), _ptr(Y), _ptr(offsets), E, rows, N, K, _stream(stream)),
           "bi_grouped_gemm_bf16")
    return Y


def grouped_gemm_silu_bf16(X, W, offsets, act=None, stream=None):
    """MoE gate_up with SiLU-mul fused: act[r] = silu(X[r] Wg[e]^T) * (X[r] Wu[e]^T),
    gate and up rounded to bf16 first, for rows r in [offsets[e], offsets[e+1]).

    X [rows,K], W [E,2I,K] bf16 (gate rows then up rows; contiguous); offsets int32 [E+1]."""
    import torch
    _dev(X, torch.bfloat16, "X"), _dev(W, torch.bfloat16, "W"), _dev(offsets, torch.int32, "offsets")
    if not (X.is_contiguous() and W.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("X, W and offsets must be contiguous")
    E, N2, K = W.shape
    rows, I = X.shape[0], N2 // 2
    if X.shape[1] != K or offsets.numel() != E + 1 or N2 % 2:
        raise ValueError("shape mismatch")
    if act is None:
        act = torch.empty((rows, I), dtype=torch.bfloat16, device=X.device)
    _dev(act, torch.bfloat16, "act")
    if act.shape != (rows, I) or not act.is_contiguous():
        raise ValueError("act must be contiguous [rows, I]")
    _check(load().bi_grouped_gemm_silu_bf16(_ptr(X), _ptr(W), _ptr(act), _ptr(offsets), E, rows, I, K,
                                            _stream(stream)), "bi_grouped_gemm_silu_bf16")
    return act


def gemm_nvfp4(A, A_sf, B, B_sf, alpha: float, Y=None, stream=None):
    """Y[M,N] = alpha * dequant(A) dequant(B)^T, e2m1 codes packed two per byte
    (uint8 [rows, K/2]) with e4m3 block scales (uint8, interleaved 128x4 layout)."""
    import torch
    for t, n in ((A, "A"), (A_sf, "A_sf"), (B, "B"), (B_sf, "B_sf")):
        _dev(t, torch.uint8, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    M, KB = A.shape
    N = B.shape[0]
    K = KB * 2
    if B.shape[1] != KB:
        raise ValueError("A and B disagree on K")
    c4 = -(-(K // 16) // 4) * 4
    if A_sf.numel() < -(-M // 128) * 128 * c4 or B_sf.numel() < -(-N // 128) * 128 * c4:
        raise ValueError("scale buffers are smaller than the interleaved layout needs")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _dev(Y, torch.bfloat16, "Y")
    if Y.shape != (M, N) or not Y.is_contiguous():
        raise ValueError("Y must be contiguous [M, N]")
    _check(load().bi_gemm_nvfp4(_ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), float(alpha), _ptr(Y), M, N, K,
                                _stream(stream)), "bi_gemm_nvfp4")
    return Y


def quantize_nvfp4(X, global_scale: float, Q=None, Q_sf=None, stream=None):
    """NVFP4-quantise bf16 rows X [M, K] with a per-tensor global scale.

    Returns (Q uint8 [M, K/2] packed e2m1, Q_sf uint8 interleaved 128x4 scales
    for ceil(M/128)*128 rows), ready for gemm_nvfp4."""
    import torch
    _dev(X, torch.bfloat16, "X")
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be [M, K] with unit column stride")
    M, K = X.shape
    if Q is None:
        Q = torch.empty((M, K // 2), dtype=torch.uint8, device=X.device)
    if Q_sf is None:
        Q_sf = torch.zeros(-(-M // 128) * 128 * (K // 16), dtype=torch.uint8, device=X.device)
    _dev(Q, torch.uint8, "Q"), _dev(Q_sf, torch.uint8, "Q_sf")
    if Q.shape != (M, K // 2) or not Q.is_contiguous() or Q_sf.numel() < -(-M // 128) * 128 * (K // 16):
        raise ValueError("output buffers have the wrong size")
    _check(load().bi_quantize_nvfp4(_ptr(X), X.stride(0), float(global_scale), _ptr(Q), _ptr(Q_sf), M, K,
                                    _stream(stream)), "bi_quantize_nvfp4")
    return Q, Q_sf


def moe_topk_softmax(logits, k: int, renormalize: bool = True, stream=None):
    """Router: (topk_ids int32 [T, k], topk_weights float32 [T, k]) from float32 logits [T, E]."""
    import torch
    _dev(logits, torch.float32, "logits")
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be contiguous [T, E]")
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(load().bi_moe_topk_softmax(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(ids), _ptr(w),
                                      _stream(stream)), "bi_moe_topk_softmax")
    return ids, w


def moe_align(topk_ids, E: int, stream=None):
    """(expert_offsets int32 [E+1], row_token int32 [T*k], pos int32 [T, k])."""
    import torch
    _dev(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    off = torch.empty(E + 1, dtype=torch.int32, device=topk_ids.device)
    row_token = torch.empty(T * k, dtype=torch.int32, device=topk_ids.device)
    pos = torch.empty((T, k), dtype=torch.int32, device=topk_ids.device)
    _check(load().bi_moe_align(_ptr(topk_ids.contiguous()), T, k, E, _ptr(off), _ptr(row_token), _ptr(pos),
                               _stream(stream)), "bi_moe_align")
    return off, row_token, pos


def moe_gather(hidden, row_token, out=None, stream=None):
    """X_sorted[r] = hidden[row_token[r]]."""
    import torch
    _dev(hidden, torch.bfloat16, "hidden"), _dev(row_token, torch.int32, "row_token")
    T, H = hidden.shape
    rows = row_token.numel()
    if out is None:
        out = torch.empty((rows, H), dtype=torch.bfloat16, device=hidden.device)
    _check(load().bi_moe_gather(_ptr(hidden), T, H, _ptr(row_token), rows, _ptr(out), _stream(stream)),
           "bi_moe_gather")
    return out


def silu_mul(gate_up, out=None, stream=None):
    """act = silu(gate) * up for bf16 rows [gate | up]."""
    import torch
    _dev(gate_up, torch.bfloat16, "gate_up")
    rows, I2 = gate_up.shape
    if out is None:
        out = torch.empty((rows, I2 // 2), dtype=torch.bfloat16, device=gate_up.device)
    _check(load().bi_silu_mul(_ptr(gate_up), rows, I2 // 2, _ptr(out), _stream(stream)), "bi_silu_mul")
    return out


def moe_combine(Y_sorted, pos, topk_weights, out=None, stream=None):
    """out[t] = sum_i w[t, i] * Y_sorted[pos[t, i]] in rank order (fp32), bf16."""
    import torch
    _dev(Y_sorted, torch.bfloat16, "Y_sorted"), _dev(pos, torch.int32, "pos")
    _dev(topk_weights, torch.float32, "topk_weights")
    rows, H = Y_sorted.shape
    T, k = pos.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=Y_sorted.device)
    _check(load().bi_moe_combine(_ptr(Y_sorted), rows, _ptr(pos), _ptr(topk_weights), T, k, H, _ptr(out),
                                 _stream(stream)), "bi_moe_combine")
    return out


def rmsnorm(x, w, eps: float, residual=None, out=None, stream=None):
    """out = bf16(h / sqrt(mean(h^2) + eps) * w), h = bf16(x + residual) (written
    back to residual) or x. x, residual, out contiguous bf16 [M, H]; w bf16 [H]."""
    import torch
    _dev(x, torch.bfloat16, "x"), _dev(w, torch.bfloat16, "w")
    if not x.is_contiguous() or not w.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be contiguous [M, H]; w contiguous [H]")
    M, H = x.shape
    if w.numel() != H:
        raise ValueError("w must have H elements")
    if residual is not None:
        _dev(residual, torch.bfloat16, "residual")
        if residual.shape != x.shape or not residual.is_contiguous():
            raise ValueError("residual must be contiguous [M, H]")
    if out is None:
        out = torch.empty_like(x)
    _dev(out, torch.bfloat16, "out")
    if out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be contiguous [M, H]")
    _check(load().bi_rmsnorm(_ptr(x), _ptr(residual) if residual is not None else None, _ptr(w), _ptr(out), M, H,
                             float(eps), _stream(stream)), "bi_rmsnorm")
    return out


def rank_sum_rmsnorm(parts, w, eps: float, residual=None, sum_out=None, out=None, stream=None):
    """Deterministic all-reduce + RMSNorm over a list of R ranks' partial rows
    (bf16 [M, H] CUDA tensors on this GPU), summed in list (rank) order."""
    import torch
    R = len(parts)
    if R < 1:
        raise ValueError("need at least one rank")
    for r, t in enumerate(parts):
        _dev(t, torch.bfloat16, f"parts[{r}]")
        if t.shape != parts[0].shape or not t.is_contiguous():
            raise ValueError("all parts must be contiguous and the same shape")
    M, H = parts[0].shape
    _dev(w, torch.bfloat16, "w")
    if out is None:
        out = torch.empty_like(parts[0])
    ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() for t in parts])
    _check(load().bi_rank_sum_rmsnorm(ptrs, R, _ptr(residual) if residual is not None else None, _ptr(w),
                                      _ptr(sum_out) if sum_out is not None else None, _ptr(out), M, H, float(eps),
                                      _stream(stream)), "bi_rank_sum_rmsnorm")
    return out


def attention_decode_workspace_size(B: int, Hq: int, max_seq_len: int) -> int:
    return int(load().bi_attention_decode_workspace_size(B, Hq, max_seq_len))


def attention_decode(Q, K_cache, V_cache, block_table, seq_lens, max_seq_len: int, scale: float,
                     workspace=None, O=None, stream=None):
    """Batch-invariant decode attention over a paged KV cache (see bi.h).

    Q bf16 [B, Hq, 128]; K_cache, V_cache bf16 [blocks, block_size, Hkv, 128];
    block_table int32 [B, max_blocks]; seq_lens int32 [B]. The workspace
    (uint8, device) is allocated with torch if not given."""
    import torch
    _dev(Q, torch.bfloat16, "Q"), _dev(K_cache, torch.bfloat16, "K_cache"), _dev(V_cache, torch.bfloat16, "V_cache")
    _dev(block_table, torch.int32, "block_table"), _dev(seq_lens, torch.int32, "seq_lens")
    for t, n in ((Q, "Q"), (K_cache, "K_cache"), (V_cache, "V_cache"), (block_table, "block_table")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, D = Q.shape
    nblk, bs, Hkv, D2 = K_cache.shape
    if D2 != D or V_cache.shape != K_cache.shape or block_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("shape mismatch")
    need = attention_decode_workspace_size(B, Hq, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=Q.device)
    if O is None:
        O = torch.empty_like(Q)
    _check(load().bi_attention_decode(_ptr(Q), _ptr(K_cache), _ptr(V_cache), _ptr(block_table), block_table.shape[1],
                                      nblk, _ptr(seq_lens), B, Hq, Hkv, D, bs, max_seq_len, float(scale),
                                      _ptr(workspace), workspace.numel(), _ptr(O), _stream(stream)),
           "bi_attention_decode")
    return O


def attention_extend(Q, cu_q, K_cache, V_cache, block_table, seq_lens, max_seq_len: int, max_q_len: int,
                     scale: float, O=None, stream=None):
    """Batch-invariant causal extend (prefill) attention over a paged KV cache (see bi.h).

    Q bf16 [total_q, Hq, 128] (each sequence's new tokens, in sequence order);
    cu_q int32 [B+1]; K_cache, V_cache bf16 [blocks, block_size, Hkv, 128];
    block_table int32 [B, max_blocks]; seq_lens int32 [B] (new tokens included)."""
    import torch
    _dev(Q, torch.bfloat16, "Q"), _dev(K_cache, torch.bfloat16, "K_cache"), _dev(V_cache, torch.bfloat16, "V_cache")
    _dev(cu_q, torch.int32, "cu_q"), _dev(block_table, torch.int32, "block_table"), _dev(seq_lens, torch.int32, "seq_lens")
    for t, n in ((Q, "Q"), (K_cache, "K_cache"), (V_cache, "V_cache"), (block_table, "block_table"), (cu_q, "cu_q")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    T, Hq, D = Q.shape
    nblk, bs, Hkv, D2 = K_cache.shape
    B = seq_lens.numel()
    if D2 != D or V_cache.shape != K_cache.shape or block_table.shape[0] != B or cu_q.numel() != B + 1:
        raise ValueError("shape mismatch")
    if O is None:
        O = torch.empty_like(Q)
    _check(load().bi_attention_extend(_ptr(Q), _ptr(cu_q), T, _ptr(K_cache), _ptr(V_cache), _ptr(block_table),
                                      block_table.shape[1], nblk, _ptr(seq_lens), B, Hq, Hkv, D, bs, max_seq_len,
                                      max_q_len, float(scale), _ptr(O), _stream(stream)), "bi_attention_extend")
    return O


def plan(op: int, M: int, N: int, K: int, num_sms: int = 0) -> dict:
    """Launch plan for these sizes (num_sms=0: the current device's SM count)."""
    p = Plan()
    _check(load().bi_plan(op, M, N, K, num_sms, ctypes.byref(p)), "bi_plan")
    return p.as_dict()


def debug_build() -> bool:
    """True when the loaded library is the bounds-checked debug build."""
    return bool(load().bi_debug_build())


def last_bounds_line() -> int:
    """Source line of the failed bounds check the last device_status() reported (0 if none)."""
    return int(load().bi_last_bounds_line())


def check_bounds(index: int, limit: int, stream=None) -> None:
    """Write element `index` of a library-owned 64-element array under a
    bounds check against `limit` (debug build: index >= limit is skipped and
    recorded; device_status() then returns BI_ERR_BOUNDS)."""
    _check(load().bi_check_bounds(index, limit, _stream(stream)), "bi_check_bounds")


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load().bi_device_status(_stream(stream)))


def check_wait_timeout(limit_us: int, stream=None):
    """Launch the bounded-wait check kernel (see bi.h)."""
    _check(load().bi_check_wait_timeout(limit_us, _stream(stream)), "bi_check_wait_timeout")
