"""bi_attention_extend on the GPU: causal extend (prefill) attention over a
paged KV cache. Parity with the fp64 oracle, and bit-exact invariance: a new
token's output equals bi_attention_decode's output for the sequence cut after
that token, whatever the prefill is split into, and whatever other sequences
share the call (batch-invariant attention backends are on the vLLM
batch-invariance tracking issue's TODO list). Qwen3-8B heads: 32 query heads,
8 KV heads, head_dim 128; other GQA groups at the end."""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_rel, bits_of, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
HQ, HKV, D, BS = 32, 8, 128, 16
SCALE = 1.0 / np.sqrt(D)
RTOL, ATOL = 1e-2, 2e-3          # the decode attention tolerance


def make(lens, qlens, seed, hq=HQ, hkv=HKV):
    lens = np.asarray(lens, dtype=np.int32)
    nb = int(-(-lens.max() // BS))
    blocks = len(lens) * nb + 3
    K = syn.to_bf16_bits(syn.normal_rows(seed, 0, blocks * BS, hkv * D)).reshape(blocks, BS, hkv, D)
    V = syn.to_bf16_bits(syn.normal_rows(seed, 1, blocks * BS, hkv * D)).reshape(blocks, BS, hkv, D)
    table = syn.rng(seed, 2).permutation(blocks)[: len(lens) * nb].astype(np.int32).reshape(len(lens), nb)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    Q = syn.to_bf16_bits(syn.normal_rows(seed, 3, int(cu[-1]) * hq, D)).reshape(int(cu[-1]), hq, D)
    return Q, cu, K, V, table, lens


def extend(bi, Q, cu, K, V, table, lens, max_len=None, max_q=None):
    qlens = np.diff(cu)
    return bits_of(bi.attention_extend(to_dev_bf16(Q), to_dev(cu), to_dev_bf16(K), to_dev_bf16(V), to_dev(table),
                                       to_dev(lens), int(max_len or lens.max()), int(max_q or max(1, qlens.max())),
                                       SCALE))


@pytest.mark.parametrize("lens,qlens", [([40, 300, 129], [40, 17, 1]),         # whole prompt, a piece, decode
                                        ([128, 257, 513], [128, 129, 200]),   # chunk boundaries 127/128/129
                                        ([1, 64, 33], [1, 5, 33])])
def test_parity(bi, lens, qlens):
    Q, cu, K, V, table, lens = make(lens, qlens, seed=sum(lens))
    got = syn.bf16_bits_to_f32(extend(bi, Q, cu, K, V, table, lens)).astype(np.float64)
    ref = oracle.attention_extend(Q, cu, K, V, table, lens, SCALE)
    assert_close_rel(got, ref, RTOL, ATOL, f"lens={list(lens)} qlens={qlens}")
    assert bi.device_status() == bi.BI_OK


def test_token_equals_decode_of_the_cut_sequence(bi):
    """Token i of the prefill gives exactly the bits bi_attention_decode gives
    for its query over the sequence cut after it (every position class: first
    chunk, chunk edges 127/128/129, the last token)."""
    L, q = 400, 300
    Q, cu, K, V, table, lens = make([L], [q], seed=7)
    full = extend(bi, Q, cu, K, V, table, lens)
    base = L - q
    for i in (0, 1, 27, 28, 29, 100, 155, 156, 157, 250, q - 1):
        pos = base + i
        one = bits_of(bi.attention_decode(to_dev_bf16(Q[i:i + 1]), to_dev_bf16(K), to_dev_bf16(V), to_dev(table),
                                          to_dev(np.array([pos + 1], np.int32)), L, SCALE))
        assert np.array_equal(one[0], full[i]), f"token {i} (position {pos}) differs from decode"


def test_prefill_split_any_way_gives_the_same_bits(bi):
    """300 new tokens in one call, or in pieces of 100, 137 and 63 tokens
    (each piece sees the cache up to its own last token)."""
    L, q = 350, 300
    Q, cu, K, V, table, lens = make([L], [q], seed=9)
    whole = extend(bi, Q, cu, K, V, table, lens)
    base, at, parts = L - q, 0, []
    for n in (100, 137, 63):
        cu_p = np.array([0, n], np.int32)
        lens_p = np.array([base + at + n], np.int32)
        parts.append(extend(bi, Q[at:at + n], cu_p, K, V, table, lens_p, max_len=L))
        at += n
    assert np.array_equal(np.concatenate(parts), whole)


def test_sequence_alone_in_other_batches_and_repeated(bi):
    lens, qlens = [90, 300, 17, 260], [90, 45, 17, 1]
    Q, cu, K, V, table, lens = make(lens, qlens, seed=11)
    full = extend(bi, Q, cu, K, V, table, lens)
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        one = extend(bi, Q[a:e], np.array([0, e - a], np.int32), K, V, table[b:b + 1], lens[b:b + 1],
                     max_len=int(lens.max()), max_q=int(np.diff(cu).max()))
        assert np.array_equal(one, full[a:e]), f"sequence {b} alone differs"
    # reversed order of the sequences
    order = [3, 2, 1, 0]
    Qr = np.concatenate([Q[cu[b]:cu[b + 1]] for b in order])
    cur = np.concatenate([[0], np.cumsum([qlens[b] for b in order])]).astype(np.int32)
    rev = extend(bi, Qr, cur, K, V, table[order], lens[order])
    at = 0
    for b in order:
        n = qlens[b]
        assert np.array_equal(rev[at:at + n], full[cu[b]:cu[b + 1]])
        at += n
    outs = {extend(bi, Q, cu, K, V, table, lens).tobytes() for _ in range(8)}
    assert len(outs) == 1
    assert bi.device_status() == bi.BI_OK


def test_empty_sequences_and_bad_lengths(bi):
    import torch
    Q, cu, K, V, table, lens = make([50, 70, 20], [10, 0, 20], seed=13)
    got = syn.bf16_bits_to_f32(extend(bi, Q, cu, K, V, table, lens)).astype(np.float64)
    ref = oracle.attention_extend(Q, cu, K, V, table, lens, SCALE)
    assert_close_rel(got, ref, RTOL, ATOL, "with an empty sequence")
    assert bi.device_status() == bi.BI_OK
    bad = lens.copy()
    bad[2] = 5                                   # 20 new tokens but 5 cached
    extend(bi, Q, cu, K, V, table, bad)
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_ERR_INVALID_ARG


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 4)])
def test_group_sizes(bi, hq, hkv):
    """GQA groups 1, 2, 8: parity, and tokens equal their decode."""
    lens, qlens = [150, 40], [150, 7]
    Q, cu, K, V, table, lens = make(lens, qlens, seed=20 + hq, hq=hq, hkv=hkv)
    full = extend(bi, Q, cu, K, V, table, lens)
    ref = oracle.attention_extend(Q, cu, K, V, table, lens, SCALE)
    assert_close_rel(syn.bf16_bits_to_f32(full).astype(np.float64), ref, RTOL, ATOL, f"Hq={hq} Hkv={hkv}")
    for t, pos in ((0, 0), (127, 127), (149, 149)):
        one = bits_of(bi.attention_decode(to_dev_bf16(Q[t:t + 1]), to_dev_bf16(K), to_dev_bf16(V),
                                          to_dev(table[:1]), to_dev(np.array([pos + 1], np.int32)), 150, SCALE))
        assert np.array_equal(one[0], full[t]), f"Hq={hq} Hkv={hkv}: token {t}"
    assert bi.device_status() == bi.BI_OK


@pytest.mark.parametrize("bs", [1, 24, 256])
def test_block_sizes(bi, bs):
    """The same cache in blocks of 1, 24 or 256 tokens gives the same bits as
    in blocks of 16, and each token still equals its decode."""
    lens, qlens = [300, 150], [300, 20]
    Q, cu, K, V, table, lens = make(lens, qlens, seed=70)
    base = extend(bi, Q, cu, K, V, table, lens)
    B, L = len(lens), int(lens.max())
    nb = -(-L // bs)
    blocks = B * nb + 2
    K2 = np.zeros((blocks, bs, HKV, D), K.dtype)
    V2 = np.zeros_like(K2)
    t2 = syn.rng(71, bs).permutation(blocks)[: B * nb].astype(np.int32).reshape(B, nb)
    for b in range(B):
        for j in range(int(lens[b])):
            K2[t2[b, j // bs], j % bs] = K[table[b, j // BS], j % BS]
            V2[t2[b, j // bs], j % bs] = V[table[b, j // BS], j % BS]
    got = extend(bi, Q, cu, K2, V2, t2, lens)
    assert np.array_equal(got, base), f"block size {bs} changed the bits"
    for i in (0, 127, 299):
        one = bits_of(bi.attention_decode(to_dev_bf16(Q[i:i + 1]), to_dev_bf16(K2), to_dev_bf16(V2),
                                          to_dev(t2[:1]), to_dev(np.array([i + 1], np.int32)), L, SCALE))
        assert np.array_equal(one[0], got[i]), f"bs={bs}: token {i} differs from decode"
    assert bi.device_status() == bi.BI_OK


def test_parity_at_the_bench_size_sampled(bi):
    """The size the bench times: one 4096-token prefill over its 4096 cached
    tokens (every query tile of the grid), Qwen3-8B heads. Sampled tokens
    at chunk edges are checked against the oracle's decode of the sequence
    cut after each."""
    import torch
    L = 4096
    nb = L // BS
    g = torch.Generator(device="cuda").manual_seed(6)
    K = torch.randn((nb, BS, HKV, D), device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn((nb, BS, HKV, D), device="cuda", generator=g).to(torch.bfloat16)
    table = torch.randperm(nb, device="cuda", generator=g).to(torch.int32).view(1, nb)
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    Q = torch.randn((L, HQ, D), device="cuda", generator=g).to(torch.bfloat16)
    got = bits_of(bi.attention_extend(Q, cu, K, V, table, lens, L, L, SCALE))
    assert bi.device_status() == bi.BI_OK
    Kb, Vb, tb = bits_of(K), bits_of(V), table.cpu().numpy()
    for i in [0, 31, 127, 128, 1000, 2049, 4095]:
        ref = oracle.attention_decode(bits_of(Q[i:i + 1]), Kb, Vb, tb, np.array([i + 1], dtype=np.int32), SCALE)
        assert_close_rel(syn.bf16_bits_to_f32(got[i:i + 1]).astype(np.float64), ref, RTOL, ATOL, f"token {i}")
