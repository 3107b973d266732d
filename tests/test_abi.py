"""The C ABI: the library loads, exports every symbol bi.h declares, plans on
the host, and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


@pytest.fixture(scope="module")
def lib():
    from invariant_deterministic_bi_gb300 import _build
    _build.build()
    import invariant_deterministic_bi_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:BI_API\s+)?(?:bi_status|const char \*|int32_t|int64_t)\s*(bi_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ["bi_gemm_bf16", "bi_grouped_gemm_bf16", "bi_grouped_gemm_silu_bf16", "bi_gemm_nvfp4", "bi_rmsnorm", "bi_plan", "bi_quantize_nvfp4", "bi_moe_topk_softmax", "bi_moe_align", "bi_moe_gather", "bi_silu_mul", "bi_moe_combine", "bi_rank_sum_rmsnorm", "bi_attention_decode", "bi_attention_decode_workspace_size", "bi_attention_extend",
              "bi_device_status", "bi_status_string", "bi_version", "bi_check_wait_timeout"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = lib.load()
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, re.M))
    for n in declared_functions():
        assert hasattr(so, n), n
        assert n in exported, n
    # nothing but the C ABI is exported from our own code
    ours = {s for s in exported if s.startswith("bi_") or s.startswith("_ZN2bi")}
    assert ours == set(declared_functions())


def test_debug_library_builds_and_exports_the_same_calls(lib):
    """libbi_debug.so (bounds-checked kernels) builds from the same sources and
    exports exactly the calls bi.h declares; it says it is the debug build."""
    from invariant_deterministic_bi_gb300 import _build
    path = _build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, re.M))
    assert {s for s in exported if s.startswith("bi_") or s.startswith("_ZN2bi")} == set(declared_functions())
    dbg = ctypes.CDLL(path)
    assert dbg.bi_debug_build() == 1
    assert lib.load().bi_debug_build() == 0
    assert dbg.bi_check_bounds(70, 10, None) == 1 and dbg.bi_check_bounds(5, 65, None) == 1   # argument checks


def test_status_strings(lib):
    assert lib.status_string(lib.BI_OK) == "BI_OK"
    assert lib.status_string(lib.BI_ERR_TIMEOUT) == "BI_ERR_TIMEOUT"
    assert lib.status_string(lib.BI_ERR_BOUNDS) == "BI_ERR_BOUNDS"
    assert lib.version() >= 100


def _plan(lib, op, M, N, K):
    return lib.plan(op, M, N, K, num_sms=152)


@pytest.mark.parametrize("N,K", [(512, 256), (6144, 4096), (24576, 4096), (4096, 12288), (264, 72)])
def test_gemm_plan_independent_of_M(lib, N, K):
    keys = ["block_m", "block_n", "block_k", "mma_m", "mma_n", "mma_k", "k_steps", "split_k", "stages",
            "threads", "smem_bytes", "tiles_n"]
    base = _plan(lib, lib.OP_GEMM_BF16, 1, N, K)
    for M in [1, 2, 7, 64, 127, 128, 129, 513, 4096, 8192, 65536]:
        p = _plan(lib, lib.OP_GEMM_BF16, M, N, K)
        assert {k: p[k] for k in keys} == {k: base[k] for k in keys}
        assert p["tiles_m"] == -(-M // p["block_m"])
        assert p["grid"] >= 2 and p["grid"] % 2 == 0             # CTA pairs
        if M > 256 or p["split_k"] == 1:                          # one pair per tile, persistent
            assert p["grid"] <= 152
        else:                                                     # one cluster of split_k pairs per column tile
            assert p["grid"] == 2 * p["split_k"] * p["tiles_n"]
    assert base["k_steps"] == -(-K // 64)
    # the K reduction's segments are fixed by (N, K): each at least 16 steps of 64
    assert 1 <= base["split_k"] <= 4 and (base["split_k"] == 1 or base["k_steps"] // base["split_k"] >= 16)


def test_gemm_segments_for_the_qwen3_layers(lib):
    """The fixed K segments of the Qwen3-8B linears and of the small config."""
    seg = lambda N, K: _plan(lib, lib.OP_GEMM_BF16, 1, N, K)["split_k"]
    assert (seg(6144, 4096), seg(24576, 4096), seg(4096, 12288)) == (2, 1, 3)
    assert seg(512, 256) == 1 and seg(2048, 768) == 1


def test_grouped_and_nvfp4_and_rmsnorm_plans_independent_of_M(lib):
    for op, N, K in [(lib.OP_GROUPED_GEMM_BF16, 1536, 2048), (lib.OP_GROUPED_GEMM_BF16, 2048, 768),
                     (lib.OP_GROUPED_GEMM_SILU_BF16, 768, 2048),
                     (lib.OP_GEMM_NVFP4, 14336, 4096), (lib.OP_RMSNORM, 4096, 0)]:
        ps = [_plan(lib, op, M, N, K) for M in [1, 3, 128, 4097, 16384]]
        for p in ps:
            for k in ["block_n", "block_k", "mma_m", "mma_n", "mma_k", "k_steps", "split_k", "reduce_tree"]:
                assert p[k] == ps[0][k], (op, k)


def test_fused_silu_plan_matches_gate_up_plan(lib):
    """The fused gate_up + SiLU-mul runs the gate_up product's tiles: same plan as N = 2I."""
    p = _plan(lib, lib.OP_GROUPED_GEMM_SILU_BF16, 4096, 768, 2048)
    q = _plan(lib, lib.OP_GROUPED_GEMM_BF16, 4096, 1536, 2048)
    assert p["op"] == lib.OP_GROUPED_GEMM_SILU_BF16
    assert {k: p[k] for k in p if k != "op"} == {k: q[k] for k in q if k != "op"}


def test_rmsnorm_plan_tree(lib):
    p = _plan(lib, lib.OP_RMSNORM, 16384, 4096, 0)
    assert p["reduce_tree"] == 32 and p["threads"] == 128 and p["block_m"] == 1 and p["grid"] == 16384
    assert _plan(lib, lib.OP_RMSNORM, 5, 65536, 0)["threads"] == 512


FAKE = 0x10000   # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,want", [
    ((FAKE, 256, FAKE, 256, FAKE, 512, -1, 512, 256), 1),          # M < 0
    ((FAKE, 256, FAKE, 256, FAKE, 512, 4, 512, 0), 1),             # K == 0
    ((None, 256, FAKE, 256, FAKE, 512, 4, 512, 256), 1),           # null X
    ((FAKE, 100, FAKE, 256, FAKE, 512, 4, 512, 256), 1),           # ldx < K
    ((FAKE, 256, FAKE, 256, FAKE, 512, 4, 512, 250), 2),           # K % 8
    ((FAKE, 256, FAKE, 256, FAKE, 516, 4, 516, 256), 2),           # N % 8
    ((FAKE + 8, 256, FAKE, 256, FAKE, 512, 4, 512, 256), 3),       # misaligned X
    ((FAKE, 260, FAKE, 256, FAKE, 512, 4, 512, 256), 3),           # ldx row stride not 16-byte
])
def test_gemm_bf16_rejects_bad_arguments(lib, args, want):
    so = lib.load()
    assert so.bi_gemm_bf16(*args, None) == want


def test_empty_work_is_ok_without_launch(lib):
    so = lib.load()
    assert so.bi_gemm_bf16(FAKE, 256, FAKE, 256, FAKE, 512, 0, 512, 256, None) == 0
    assert so.bi_grouped_gemm_bf16(FAKE, FAKE, FAKE, FAKE, 128, 0, 1536, 2048, None) == 0
    assert so.bi_gemm_nvfp4(FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), FAKE, 0, 64, 128, None) == 0
    assert so.bi_rmsnorm(FAKE, None, FAKE, FAKE, 0, 4096, ctypes.c_float(1e-6), None) == 0


def test_other_calls_reject_bad_arguments(lib):
    so = lib.load()
    f = ctypes.c_float
    assert so.bi_grouped_gemm_bf16(FAKE, FAKE, FAKE, FAKE, 0, 8, 64, 64, None) == 1        # E < 1
    assert so.bi_grouped_gemm_bf16(FAKE, FAKE, FAKE, FAKE, 2000, 8, 64, 64, None) == 1     # E > 1024
    assert so.bi_grouped_gemm_bf16(FAKE, FAKE, FAKE, FAKE + 2, 4, 8, 64, 64, None) == 3    # offsets align
    assert so.bi_grouped_gemm_silu_bf16(FAKE, FAKE, FAKE, FAKE, 0, 8, 768, 64, None) == 1   # E < 1
    assert so.bi_grouped_gemm_silu_bf16(FAKE, FAKE, FAKE, FAKE, 4, 8, 96, 64, None) == 2    # I % 128
    assert so.bi_grouped_gemm_silu_bf16(FAKE, FAKE, FAKE, FAKE, 4, 8, 768, 60, None) == 2   # K % 8
    assert so.bi_grouped_gemm_silu_bf16(FAKE, FAKE, FAKE + 8, FAKE, 4, 8, 768, 64, None) == 3   # act align
    assert so.bi_grouped_gemm_silu_bf16(FAKE, FAKE, FAKE, FAKE, 4, 0, 768, 64, None) == 0   # no rows
    assert so.bi_gemm_nvfp4(FAKE, FAKE, FAKE, FAKE, f(1.0), FAKE, 4, 64, 96, None) == 2    # K % 64
    assert so.bi_gemm_nvfp4(FAKE, FAKE + 4, FAKE, FAKE, f(1.0), FAKE, 4, 64, 128, None) == 3
    assert so.bi_rmsnorm(FAKE, None, FAKE, FAKE, 4, 4, f(1e-6), None) == 1                 # H < 8
    assert so.bi_rmsnorm(FAKE, None, FAKE, FAKE, 4, 4100, f(1e-6), None) == 2              # H % 8
    assert so.bi_rmsnorm(FAKE, None, FAKE, FAKE, 4, 4096, f(-1.0), None) == 1              # eps < 0
    assert so.bi_rmsnorm(FAKE, None, FAKE, FAKE, 1 << 31, 4096, f(1e-6), None) == 1        # M >= 2^31 - 1
    assert so.bi_rmsnorm(FAKE, FAKE + 8, FAKE, FAKE, 4, 4096, f(1e-6), None) == 3          # residual align
    assert so.bi_quantize_nvfp4(FAKE, 128, f(1.0), FAKE, FAKE, 4, 96, None) == 2           # K % 64
    assert so.bi_quantize_nvfp4(FAKE, 128, f(0.0), FAKE, FAKE, 4, 128, None) == 1          # scale <= 0
    assert so.bi_quantize_nvfp4(FAKE, 128, f(2.0 ** 65), FAKE, FAKE, 4, 128, None) == 1    # scale > 2^64
    assert so.bi_quantize_nvfp4(FAKE, 100, f(1.0), FAKE, FAKE, 4, 128, None) == 1          # ldx < K
    assert so.bi_quantize_nvfp4(FAKE, 136, f(1.0), FAKE + 8, FAKE, 4, 128, None) == 3      # Q align
    assert so.bi_quantize_nvfp4(FAKE, 128, f(1.0), FAKE, FAKE, 0, 128, None) == 0          # empty
    assert so.bi_moe_topk_softmax(FAKE, 4, 128, 0, 1, FAKE, FAKE, None) == 1             # k < 1
    assert so.bi_moe_topk_softmax(FAKE, 4, 2000, 8, 1, FAKE, FAKE, None) == 1            # E > 1024
    assert so.bi_moe_topk_softmax(FAKE, 4, 4, 8, 1, FAKE, FAKE, None) == 1               # k > E
    assert so.bi_moe_topk_softmax(FAKE, 0, 128, 8, 1, FAKE, FAKE, None) == 0             # empty
    assert so.bi_moe_align(FAKE + 2, 4, 8, 128, FAKE, FAKE, FAKE, None) == 3
    assert so.bi_moe_align(FAKE, 1 << 61, 8, 128, FAKE, FAKE, FAKE, None) == 1          # T * k past 2^31 - 1
    assert so.bi_moe_gather(FAKE, 4, 100, FAKE, 8, FAKE, None) == 2                      # H % 8
    assert so.bi_silu_mul(FAKE, 4, 12, FAKE, None) == 2                                  # I % 8
    assert so.bi_moe_combine(FAKE, 8, FAKE, FAKE, 4, 0, 64, FAKE, None) == 1              # k < 1
    ptrs2 = (ctypes.c_void_p * 2)(FAKE, FAKE + 8)
    assert so.bi_rank_sum_rmsnorm(ptrs2, 2, None, FAKE, None, FAKE, 4, 4096, f(1e-6), None) == 3  # part align
    assert so.bi_rank_sum_rmsnorm(ptrs2, 0, None, FAKE, None, FAKE, 4, 4096, f(1e-6), None) == 1  # R < 1
    assert so.bi_rank_sum_rmsnorm(ptrs2, 17, None, FAKE, None, FAKE, 4, 4096, f(1e-6), None) == 1  # R > 16
    A = so.bi_attention_decode
    ok_args = lambda **kw: dict(dict(Q=FAKE, K=FAKE, V=FAKE, table=FAKE, mb=8, nb=64, lens=FAKE, B=4, Hq=32, Hkv=8,
                                     D=128, bs=16, L=128, scale=f(0.1), ws=FAKE, wsb=1 << 30, O=FAKE), **kw)
    call = lambda a: A(a["Q"], a["K"], a["V"], a["table"], a["mb"], a["nb"], a["lens"], a["B"], a["Hq"], a["Hkv"],
                       a["D"], a["bs"], a["L"], a["scale"], a["ws"], a["wsb"], a["O"], None)
    assert call(ok_args(D=64)) == 2                 # head_dim != 128
    assert call(ok_args(Hkv=3)) == 2                # Hq % Hkv
    assert call(ok_args(Hq=48, Hkv=4)) == 2         # group of 12
    assert call(ok_args(wsb=100)) == 1              # workspace too small
    assert call(ok_args(Q=FAKE + 8)) == 3
    assert call(ok_args(B=0)) == 0
    assert so.bi_attention_decode_workspace_size(4, 32, 300) == 4 * 32 * 3 * 130 * 4   # ceil(300 / 128) chunks
    # the longest sequence bound, and sizes past int64_t, give -1 and refuse the calls
    assert so.bi_attention_decode_workspace_size(1, 1, 1 << 30) == (1 << 23) * 130 * 4
    assert so.bi_attention_decode_workspace_size(1, 1, (1 << 30) + 1) == -1
    assert so.bi_attention_decode_workspace_size(65535, 1 << 30, 1 << 30) == -1
    assert call(ok_args(L=(1 << 30) + 1)) == 1
    assert call(ok_args(B=65535, Hq=1 << 30, Hkv=1 << 27, L=1 << 30)) == 1
    N = so.bi_attention_decode_noalloc
    assert N(FAKE, FAKE, FAKE, FAKE, 8, 64, FAKE, 65535, 1 << 30, 1 << 27, 128, 16, 1 << 30, f(0.1), FAKE,
             None) == 2
    assert so.bi_attention_extend(FAKE, FAKE, 4, FAKE, FAKE, FAKE, 8, 64, FAKE, 4, 32, 8, 128, 16, (1 << 30) + 1, 4,
                                  f(0.1), FAKE, None) == 1
    assert so.bi_check_wait_timeout(0, None) == 1
    assert so.bi_plan(99, 1, 1, 1, 152, ctypes.byref(lib.Plan())) == 1
