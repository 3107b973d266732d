"""bi_attention_decode_noalloc: decode attention for callers that cannot
allocate device memory (for example code whose host program has reserved all
device memory up front, or a latency-critical path that must not risk the
synchronisation an allocation can cause). The entry point keeps its partial
results in a fixed array the library owns. This file checks, through the C
ABI, that it returns bit for bit what bi_attention_decode returns with a
caller-provided workspace (the same kernels run on the same inputs), on two
calls in a row, that its output is within the attention tolerance of the
oracle, that the largest problem that fits the array is accepted and the next
one up refused. It is named to run last."""
import ctypes

import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_rel, bits_of, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
HQ, HKV, D, BS = 32, 8, 128, 16
SCALE = 1.0 / np.sqrt(D)
CHUNK = 128                      # tokens per split of the decode kernel
LIMIT = 16 << 20                 # BI_ATTENTION_NOALLOC_SCRATCH_BYTES
# attention tolerance: |gpu - ref| <= 1e-2 |ref| + 2e-3 (the decode attention tests use the same)
RTOL, ATOL = 1e-2, 2e-3


def cache(lens, seed):
    """A paged cache holding exactly the blocks the sequences need, in a
    seeded random order; unused table entries point at block 0."""
    lens = np.asarray(lens, dtype=np.int32)
    need = -(-lens // BS)
    blocks = int(need.sum())
    K = syn.to_bf16_bits(syn.normal_rows(seed, 0, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    V = syn.to_bf16_bits(syn.normal_rows(seed, 1, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    order = syn.rng(seed, 2).permutation(blocks).astype(np.int32)
    table = np.zeros((len(lens), int(need.max())), dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = order[at:at + n]
        at += n
    Q = syn.to_bf16_bits(syn.normal_rows(seed, 3, len(lens) * HQ, D)).reshape(len(lens), HQ, D)
    return Q, K, V, table, lens


def noalloc(lib, Qd, Kd, Vd, td, ld, B, nblocks, max_len, Od, stream):
    return lib.bi_attention_decode_noalloc(
        ctypes.c_void_p(Qd.data_ptr()), ctypes.c_void_p(Kd.data_ptr()), ctypes.c_void_p(Vd.data_ptr()),
        ctypes.c_void_p(td.data_ptr()), td.shape[1], nblocks, ctypes.c_void_p(ld.data_ptr()), B, HQ, HKV, D, BS,
        max_len, ctypes.c_float(SCALE), ctypes.c_void_p(Od.data_ptr()), stream)


def run_both(bi, lib, Q, K, V, table, lens, max_len, with_ref=True):
    """(noalloc status, noalloc output bits, workspace-entry output bits or None)."""
    import torch
    Qd, Kd, Vd, td, ld = to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev(table), to_dev(lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = bi.attention_decode(Qd, Kd, Vd, td, ld, max_len, SCALE) if with_ref else None   # caller's workspace
    Od = torch.full_like(Qd, float("nan"))
    st = noalloc(lib, Qd, Kd, Vd, td, ld, len(lens), K.shape[0], max_len, Od, stream)
    torch.cuda.synchronize()
    return st, bits_of(Od), (bits_of(ref) if with_ref else None)


def check_against_oracle(got_bits, Q, K, V, table, lens, what):
    want = oracle.attention_decode(Q, K, V, table, lens, SCALE)
    assert_close_rel(syn.bf16_bits_to_f32(got_bits).astype(np.float64), want, RTOL, ATOL, what)


def test_noalloc_matches_workspace_entry_point_twice(bi):
    lib = bi.load()
    for call, (lens, seed) in enumerate([([700, 33, 4000, 256, 1], 41), ([1, 257, 1024], 42)]):
        Q, K, V, table, lens = cache(lens, seed)
        st, got, ref = run_both(bi, lib, Q, K, V, table, lens, int(lens.max()))
        assert st == bi.BI_OK, f"call {call}: {bi.status_string(st)}"
        assert np.array_equal(got, ref), f"call {call}: differs from bi_attention_decode"
        check_against_oracle(got, Q, K, V, table, lens, f"call {call}")
    assert bi.device_status() == bi.BI_OK


def test_noalloc_largest_problem_that_fits_and_next_refused(bi):
    """B = 8 sequences of 32 query heads: up to 126 chunks of partials fit in
    the array (126 * 8 * 32 * 130 * 4 bytes = LIMIT - 4096), 127 do not."""
    lib = bi.load()
    B, fits = 8, 126 * CHUNK
    assert bi.attention_decode_workspace_size(B, HQ, fits) <= LIMIT
    assert bi.attention_decode_workspace_size(B, HQ, fits + 1) > LIMIT
    lens = [fits, 5, 300, 1, 4000, 129, 128, fits - 1]
    Q, K, V, table, lens = cache(lens, 43)
    st, got, ref = run_both(bi, lib, Q, K, V, table, lens, fits)
    assert st == bi.BI_OK, bi.status_string(st)
    assert np.array_equal(got, ref)
    check_against_oracle(got, Q, K, V, table, lens, "largest problem")
    # one more chunk of capacity is refused before anything is launched: O keeps its NaN fill
    st, got, _ = run_both(bi, lib, Q, K, V, table, lens, fits + 1, with_ref=False)
    assert st == bi.BI_ERR_UNSUPPORTED
    assert np.all((got & 0x7FFF) > 0x7F80), "a refused call wrote its output"
    assert bi.device_status() == bi.BI_OK


def test_noalloc_refuses_problems_beyond_its_array(bi):
    import torch
    lib = bi.load()
    B, max_len = 64, 4096
    assert bi.attention_decode_workspace_size(B, HQ, max_len) > LIMIT
    Qd = torch.zeros((B, HQ, D), dtype=torch.bfloat16, device="cuda")
    Kd = torch.zeros((B, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    td = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    ld = torch.ones(B, dtype=torch.int32, device="cuda")
    Od = torch.empty_like(Qd)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = noalloc(lib, Qd, Kd, Kd, td, ld, B, B, max_len, Od, stream)
    assert st == bi.BI_ERR_UNSUPPORTED
