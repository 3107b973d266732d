"""bi_attention_decode_noalloc: decode attention for callers that cannot
allocate device memory (for example code whose host program has reserved all
device memory up front, or a latency-critical path that must not risk the
synchronisation an allocation can cause). The entry point keeps its partial
results in a fixed array the library owns; this file checks, through the C
ABI, that it returns what bi_attention_decode returns with a caller-provided
workspace, on two calls in a row, and that problems too large for the array
are refused. It is named to run last."""
import ctypes

import numpy as np
import pytest

import bi_synth as syn
from util import assert_close_rel, bits_of, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
HQ, HKV, D, BS = 32, 8, 128, 16
SCALE = 1.0 / np.sqrt(D)


def cache(lens, seed):
    lens = np.asarray(lens, dtype=np.int32)
    nb = int(-(-lens.max() // BS))
    blocks = len(lens) * nb
    K = syn.to_bf16_bits(syn.normal_rows(seed, 0, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    V = syn.to_bf16_bits(syn.normal_rows(seed, 1, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    table = syn.rng(seed, 2).permutation(blocks).astype(np.int32).reshape(len(lens), nb)
    Q = syn.to_bf16_bits(syn.normal_rows(seed, 3, len(lens) * HQ, D)).reshape(len(lens), HQ, D)
    return Q, K, V, table, lens


def noalloc(lib, Qd, Kd, Vd, td, ld, B, nblocks, max_len, Od, stream):
    return lib.bi_attention_decode_noalloc(
        ctypes.c_void_p(Qd.data_ptr()), ctypes.c_void_p(Kd.data_ptr()), ctypes.c_void_p(Vd.data_ptr()),
        ctypes.c_void_p(td.data_ptr()), td.shape[1], nblocks, ctypes.c_void_p(ld.data_ptr()), B, HQ, HKV, D, BS,
        max_len, ctypes.c_float(SCALE), ctypes.c_void_p(Od.data_ptr()), stream)


def test_noalloc_matches_workspace_entry_point_twice(bi):
    import torch
    lib = bi.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (lens, seed) in enumerate([([700, 33, 4000, 256, 1], 41), ([1, 257, 1024], 42)]):
        Q, K, V, table, lens = cache(lens, seed)
        Qd, Kd, Vd, td, ld = to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev(table), to_dev(lens)
        max_len = int(lens.max())
        ref = bi.attention_decode(Qd, Kd, Vd, td, ld, max_len, SCALE)      # caller-provided workspace
        Od = torch.empty_like(Qd)
        st = noalloc(lib, Qd, Kd, Vd, td, ld, len(lens), K.shape[0], max_len, Od, stream)
        assert st == bi.BI_OK, f"call {call}: {bi.status_string(st)}"
        torch.cuda.synchronize()
        got = syn.bf16_bits_to_f32(bits_of(Od)).astype(np.float64)
        want = syn.bf16_bits_to_f32(bits_of(ref)).astype(np.float64)
        assert_close_rel(got, want, 1e-2, 2e-3, f"call {call}")
    assert bi.device_status() == bi.BI_OK


def test_noalloc_refuses_problems_beyond_its_array(bi):
    import torch
    lib = bi.load()
    limit = 16 << 20
    B, max_len = 64, 4096
    assert bi.attention_decode_workspace_size(B, HQ, max_len) > limit
    Qd = torch.zeros((B, HQ, D), dtype=torch.bfloat16, device="cuda")
    Kd = torch.zeros((B, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    td = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    ld = torch.ones(B, dtype=torch.int32, device="cuda")
    Od = torch.empty_like(Qd)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = noalloc(lib, Qd, Kd, Kd, td, ld, B, B, max_len, Od, stream)
    assert st == bi.BI_ERR_UNSUPPORTED
