"""bi_attention_decode on the GPU: parity with the fp64 oracle and bit-exact
batch invariance of decode attention over a paged KV cache (Qwen3-8B heads:
32 query heads, 8 KV heads, head_dim 128). Batch-invariant attention is on the
vLLM batch-invariance tracking issue's TODO list."""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_rel, bits_of, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
HQ, HKV, D, BS = 32, 8, 128, 16
SCALE = 1.0 / np.sqrt(D)


def make_cache(lens, seed=0, spare_blocks=3):
    lens = np.asarray(lens, dtype=np.int32)
    nb = int(-(-lens.max() // BS))
    blocks = len(lens) * nb + spare_blocks
    K = syn.to_bf16_bits(syn.normal_rows(seed, 0, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    V = syn.to_bf16_bits(syn.normal_rows(seed, 1, blocks * BS, HKV * D)).reshape(blocks, BS, HKV, D)
    perm = syn.rng(seed, 2).permutation(blocks)[: len(lens) * nb].astype(np.int32)
    return K, V, perm.reshape(len(lens), nb), lens


def run(bi, Q, K, V, table, lens, max_len):
    return bits_of(bi.attention_decode(to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev(table),
                                       to_dev(lens), max_len, SCALE))


@pytest.mark.parametrize("lens", [[1, 300, 1000], [127, 128, 129, 255], [256, 257, 512, 513], [4096, 7],
                                  [4097, 8192, 8193, 33]])   # the merge takes chunks in tiles of 32
def test_parity(bi, lens):
    K, V, table, lens = make_cache(lens, seed=len(lens))
    B = len(lens)
    Q = syn.to_bf16_bits(syn.normal_rows(9, 0, B * HQ, D)).reshape(B, HQ, D)
    got = syn.bf16_bits_to_f32(run(bi, Q, K, V, table, lens, int(lens.max()))).astype(np.float64)
    ref = oracle.attention_decode(Q, K, V, table, lens, SCALE)
    assert_close_rel(got, ref, 1e-2, 2e-3, f"lens={list(lens)}")
    assert bi.device_status() == bi.BI_OK


def test_single_token_sequences_return_values(bi):
    """One cached token: softmax weight 1, the output is v itself (bf16 exact)."""
    K, V, table, lens = make_cache([1, 1, 1], seed=11)
    Q = syn.to_bf16_bits(syn.normal_rows(12, 0, 3 * HQ, D)).reshape(3, HQ, D)
    got = run(bi, Q, K, V, table, lens, 64)
    for b in range(3):
        v = V[table[b, 0], 0]
        for h in range(HQ):
            assert np.array_equal(got[b, h], v[h // (HQ // HKV)])


def test_batch_invariance(bi):
    """A sequence's output is the same bits alone, in this batch, in another
    batch and after reordering; 8 identical runs give one output."""
    lens = [700, 33, 4000, 256, 1]
    K, V, table, lens = make_cache(lens, seed=21)
    B = len(lens)
    Q = syn.to_bf16_bits(syn.normal_rows(22, 0, B * HQ, D)).reshape(B, HQ, D)
    full = run(bi, Q, K, V, table, lens, 4096)
    for b in range(B):
        one = run(bi, Q[b:b + 1], K, V, table[b:b + 1], lens[b:b + 1], 4096)
        assert np.array_equal(one[0], full[b]), f"sequence {b} alone differs"
        other = run(bi, Q[b:b + 1], K, V, table[b:b + 1], lens[b:b + 1], int(lens[b]))
        assert np.array_equal(other[0], full[b]), f"sequence {b}: max_seq_len changed its bits"
    perm = np.array([3, 0, 4, 2, 1])
    pr = run(bi, Q[perm], K, V, table[perm], lens[perm], 4096)
    assert np.array_equal(pr, full[perm])
    outs = {run(bi, Q, K, V, table, lens, 4096).tobytes() for _ in range(8)}
    assert len(outs) == 1


def test_bad_lengths_reported(bi):
    import torch
    K, V, table, lens = make_cache([10, 10], seed=31)
    Q = syn.to_bf16_bits(syn.normal_rows(32, 0, 2 * HQ, D)).reshape(2, HQ, D)
    bad = np.array([10, 0], dtype=np.int32)
    bi.attention_decode(to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev(table), to_dev(bad), 16, SCALE)
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_ERR_INVALID_ARG


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 4)])
def test_group_sizes(bi, hq, hkv):
    """GQA groups G = 1, 2, 8 (the shapes above use G = 4): parity with the
    oracle, and a sequence alone gives the same bits as in the batch."""
    lens = np.asarray([1, 129, 300], dtype=np.int32)
    nb = int(-(-lens.max() // BS))
    blocks = len(lens) * nb + 2
    K = syn.to_bf16_bits(syn.normal_rows(40 + hq, 0, blocks * BS, hkv * D)).reshape(blocks, BS, hkv, D)
    V = syn.to_bf16_bits(syn.normal_rows(40 + hq, 1, blocks * BS, hkv * D)).reshape(blocks, BS, hkv, D)
    table = syn.rng(40 + hq, 2).permutation(blocks)[: len(lens) * nb].astype(np.int32).reshape(len(lens), nb)
    Q = syn.to_bf16_bits(syn.normal_rows(41 + hq, 0, len(lens) * hq, D)).reshape(len(lens), hq, D)
    full = run(bi, Q, K, V, table, lens, 512)
    got = syn.bf16_bits_to_f32(full).astype(np.float64)
    ref = oracle.attention_decode(Q, K, V, table, lens, SCALE)
    assert_close_rel(got, ref, 1e-2, 2e-3, f"Hq={hq} Hkv={hkv}")
    for b in range(len(lens)):
        one = run(bi, Q[b:b + 1], K, V, table[b:b + 1], lens[b:b + 1], 512)
        assert np.array_equal(one[0], full[b]), f"Hq={hq} Hkv={hkv}: sequence {b} alone differs"
    assert bi.device_status() == bi.BI_OK


def relayout(K, V, table, lens, bs, seed):
    """The same sequences' K/V in a cache of block size bs (blocks in a
    seeded random order, two spare blocks)."""
    B, L = len(lens), int(lens.max())
    nb = -(-L // bs)
    blocks = B * nb + 2
    K2 = np.zeros((blocks, bs) + K.shape[2:], K.dtype)
    V2 = np.zeros_like(K2)
    t2 = syn.rng(seed, 5).permutation(blocks)[: B * nb].astype(np.int32).reshape(B, nb)
    for b in range(B):
        for j in range(int(lens[b])):
            K2[t2[b, j // bs], j % bs] = K[table[b, j // BS], j % BS]
            V2[t2[b, j // bs], j % bs] = V[table[b, j // BS], j % BS]
    return K2, V2, t2


@pytest.mark.parametrize("bs", [1, 8, 24, 128, 256])
def test_block_sizes(bi, bs):
    """Block sizes the whole-block copies tile (8, 128, 256) and ones they do
    not (1, 24): the same sequences give the same bits as with 16-token
    blocks, and parity with the oracle."""
    lens = np.asarray([300, 1, 129, 640], dtype=np.int32)
    K, V, table, lens = make_cache(lens, seed=50)
    Q = syn.to_bf16_bits(syn.normal_rows(51, 0, len(lens) * HQ, D)).reshape(len(lens), HQ, D)
    base = run(bi, Q, K, V, table, lens, 640)
    K2, V2, t2 = relayout(K, V, table, lens, bs, seed=bs)
    got = run(bi, Q, K2, V2, t2, lens, 640)
    assert np.array_equal(got, base), f"block size {bs} changed the bits"
    ref = oracle.attention_decode(Q, K2, V2, t2, lens, SCALE)
    assert_close_rel(syn.bf16_bits_to_f32(got).astype(np.float64), ref, 1e-2, 2e-3, f"bs={bs}")
    assert bi.device_status() == bi.BI_OK


@pytest.mark.parametrize("bs", [16, 24])
def test_block_outside_the_cache_reported(bi, bs):
    """A block-table entry outside the cache: its tokens are left out (score
    -inf) and the device status reports it."""
    import torch
    lens = np.asarray([200, 50], dtype=np.int32)
    K, V, table, lens = make_cache(lens, seed=60)
    K2, V2, t2 = relayout(K, V, table, lens, bs, seed=61)
    t2 = t2.copy()
    t2[0, 1] = K2.shape[0] + 7
    Q = syn.to_bf16_bits(syn.normal_rows(62, 0, 2 * HQ, D)).reshape(2, HQ, D)
    got = run(bi, Q, K2, V2, t2, lens, 256)
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_ERR_INVALID_ARG
    good = run(bi, Q[1:], K2, V2, t2[1:], lens[1:], 256)
    assert np.array_equal(got[1], good[0])
    assert np.all(np.isfinite(syn.bf16_bits_to_f32(got)))


def test_parity_at_the_bench_size_sampled(bi):
    """The size the bench times: 64 sequences of 4096 cached tokens (the
    persistent ring shape), Qwen3-8B heads, 16-token blocks in a random order;
    two sequences cut short (a partial last chunk). Six sequences are checked
    whole against the oracle, on their own blocks."""
    import torch
    B, L = 64, 4096
    nb = L // BS
    g = torch.Generator(device="cuda").manual_seed(5)
    K = torch.randn((B * nb, BS, HKV, D), device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn((B * nb, BS, HKV, D), device="cuda", generator=g).to(torch.bfloat16)
    table = torch.randperm(B * nb, device="cuda", generator=g).to(torch.int32).view(B, nb)
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    lens[3], lens[40] = 4000, 129
    Q = torch.randn((B, HQ, D), device="cuda", generator=g).to(torch.bfloat16)
    got = bits_of(bi.attention_decode(Q, K, V, table, lens, L, SCALE))
    assert bi.device_status() == bi.BI_OK
    for b in [0, 3, 17, 40, 62, 63]:
        blk = table[b].long()
        n = int(lens[b].item())
        ref = oracle.attention_decode(bits_of(Q[b:b + 1]), bits_of(K[blk]), bits_of(V[blk]),
                                      np.arange(nb, dtype=np.int32)[None], np.array([n], dtype=np.int32), SCALE)
        assert_close_rel(syn.bf16_bits_to_f32(got[b:b + 1]).astype(np.float64), ref, 1e-2, 2e-3, f"sequence {b}")
