"""The MoE layer on the GPU (routing, alignment, gather, grouped GEMMs, SiLU-mul,
combine): each step against the oracle, a full layer end to end, and the
property that matters: a token's output does not depend on the tokens it is
batched with (batch invariance, vllm-ascend guide; MoE models listed as
tested there: Qwen3-30B-A3B, whose shapes these are).
"""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, assert_close_rel, bits_of, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
E, TOPK, HID, INTER = 128, 8, 2048, 768


def logits_for(T, seed=0, ties=True):
    l = syn.normal_rows(seed, syn.TID_LOGITS, T, E)
    if ties and T > 3:
        l[1, 5] = l[1, 9] = l[1].max() + 0.5        # exact tie at the top
        l[2, 100] = l[2, 3] = l[2, 64]               # three-way tie
    return l


@pytest.mark.parametrize("T", [1, 8, 64, 512, 8192])
@pytest.mark.parametrize("renorm", [True, False])
def test_topk_softmax(bi, T, renorm):
    l = logits_for(T)
    ids, w = bi.moe_topk_softmax(to_dev(l), TOPK, renormalize=renorm)
    oids, ow = oracle.moe_topk_softmax(l, TOPK, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert_close_rel(w.cpu().numpy().astype(np.float64), ow, 2e-6, 1e-9, "weights")
    # a token alone gets the same bits
    for t in sample_rows(T, 3, seed=T):
        i1, w1 = bi.moe_topk_softmax(to_dev(l[t:t + 1]), TOPK, renormalize=renorm)
        assert np.array_equal(i1.cpu().numpy()[0], ids.cpu().numpy()[t])
        assert np.array_equal(w1.cpu().numpy()[0], w.cpu().numpy()[t])


@pytest.mark.parametrize("T", [1, 7, 16, 17, 512, 2048, 8192])   # one block up to 128 pairs, then the multi-block path
def test_align_exact(bi, T):
    ids = oracle.moe_topk_softmax(logits_for(T, seed=1), TOPK)[0]
    off, row_token, pos = bi.moe_align(to_dev(ids), E)
    o_off, o_rt, o_pos = oracle.moe_align(ids, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(row_token.cpu().numpy(), o_rt)
    assert np.array_equal(pos.cpu().numpy(), o_pos)


@pytest.mark.parametrize("E_,T,k", [(1, 100, 1), (1, 300, 1), (3, 60, 2), (3, 2000, 2), (1024, 4, 8), (1024, 16, 8),
                                     (1024, 600, 4), (1024, 3000, 8)])
def test_align_exact_expert_counts(bi, E_, T, k):
    """Any ids in [0, E): one expert, few experts, the largest E, both paths."""
    ids = np.random.default_rng(E_ * 7 + T).integers(0, E_, size=(T, k)).astype(np.int32)
    off, row_token, pos = bi.moe_align(to_dev(ids), E_)
    o_off, o_rt, o_pos = oracle.moe_align(ids, E_)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(row_token.cpu().numpy(), o_rt)
    assert np.array_equal(pos.cpu().numpy(), o_pos)


@pytest.mark.parametrize("T", [300, 3000])
def test_align_with_unaligned_ids(bi, T):
    """An id array that starts 4 bytes past a 16-byte boundary (the multi-block
    path's scalar loads at T = 3000): same result."""
    import torch
    ids = oracle.moe_topk_softmax(logits_for(T, seed=3), TOPK)[0]
    buf = torch.zeros(T * TOPK + 1, dtype=torch.int32, device="cuda")
    buf[1:] = to_dev(ids).view(-1)
    view = buf[1:].view(T, TOPK)
    assert view.data_ptr() % 16 == 4
    off, row_token, pos = bi.moe_align(view, E)
    o_off, o_rt, o_pos = oracle.moe_align(ids, E)
    assert np.array_equal(off.cpu().numpy(), o_off) and np.array_equal(pos.cpu().numpy(), o_pos)
    assert np.array_equal(row_token.cpu().numpy(), o_rt)


def test_align_rejects_bad_ids(bi):
    import torch
    ids = np.zeros((4, 2), dtype=np.int32)
    ids[2, 1] = 500
    bi.moe_align(to_dev(ids), 16)
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_ERR_INVALID_ARG


def test_gather_and_silu_mul(bi):
    T, H = 300, 2048
    hidden = syn.to_bf16_bits(syn.normal_rows(2, syn.TID_HIDDEN, T, H))
    ids = oracle.moe_topk_softmax(logits_for(T, seed=2), TOPK)[0]
    _, rt, _ = oracle.moe_align(ids, E)
    X = bits_of(bi.moe_gather(to_dev_bf16(hidden), to_dev(rt)))
    assert np.array_equal(X, hidden[rt])
    gu = syn.to_bf16_bits(syn.normal_rows(3, syn.TID_DOWN_IN, 517, 2 * INTER, std=3.0))
    act = bits_of(bi.silu_mul(to_dev_bf16(gu)))
    ref = oracle.silu_mul(gu)
    assert_close_rel(syn.bf16_bits_to_f32(act).astype(np.float64), ref, 8e-3, 1e-6, "silu_mul")


def test_combine(bi):
    T, H, rows = 257, 2048, 257 * TOPK
    Y = syn.to_bf16_bits(syn.normal_rows(4, syn.TID_DOWN_IN, rows, H))
    ids, w = oracle.moe_topk_softmax(logits_for(T, seed=4), TOPK)
    _, _, pos = oracle.moe_align(ids, E)
    w32 = w.astype(np.float32)
    out = bits_of(bi.moe_combine(to_dev_bf16(Y), to_dev(pos), to_dev(w32)))
    ref = oracle.moe_combine(Y, pos, w32.astype(np.float64))
    mag = oracle.moe_combine(Y & np.uint16(0x7FFF), pos, np.abs(w32).astype(np.float64))   # sum of |w * y|
    err = np.abs(syn.bf16_bits_to_f32(out).astype(np.float64) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6 * mag + 1e-30)


@pytest.fixture(scope="module")
def layer_weights():
    W1 = syn.moe_weights(E, 2 * INTER, HID, seed=0, tensor_id=syn.TID_W1)
    W2 = syn.moe_weights(E, HID, INTER, seed=0, tensor_id=syn.TID_W2)
    return W1, W2, to_dev_bf16(W1), to_dev_bf16(W2)


def gpu_layer(bi, hidden_bits, logits, W1d, W2d, fused=False):
    hd, ld = to_dev_bf16(hidden_bits), to_dev(logits)
    ids, w = bi.moe_topk_softmax(ld, TOPK)
    off, rt, pos = bi.moe_align(ids, E)
    X = bi.moe_gather(hd, rt)
    if fused:
        gu = None
        act = bi.grouped_gemm_silu_bf16(X, W1d, off)
    else:
        gu = bi.grouped_gemm_bf16(X, W1d, off)
        act = bi.silu_mul(gu)
    y = bi.grouped_gemm_bf16(act, W2d, off)
    return bits_of(bi.moe_combine(y, pos, w)), (bits_of(gu) if gu is not None else None)


def test_full_layer_against_oracle_and_token_invariance(bi, layer_weights):
    W1, W2, W1d, W2d = layer_weights
    T = 512
    hidden = syn.to_bf16_bits(syn.normal_rows(5, syn.TID_HIDDEN, T, HID))
    logits = logits_for(T, seed=5)
    out, _ = gpu_layer(bi, hidden, logits, W1d, W2d)
    # oracle chain, rounding to bf16 where the GPU path stores bf16
    ids, w = oracle.moe_topk_softmax(logits, TOPK)
    off, rt, pos = oracle.moe_align(ids, E)
    rows = sample_rows(T, 24, seed=6)
    for t in rows:
        mine = [pos[t, i] for i in range(TOPK)]
        ys = []
        for i, r in enumerate(mine):
            e = ids[t, i]
            gu = oracle.bf16_round_array(oracle.gemm_bf16(hidden[t:t + 1], W1[e]))
            act = oracle.bf16_round_array(oracle.silu_mul(gu))
            ys.append(oracle.bf16_round_array(oracle.gemm_bf16(act, W2[e]))[0])
        Ytok = np.stack(ys)
        ref = oracle.moe_combine(Ytok, np.arange(TOPK, dtype=np.int32)[None], w[t:t + 1].astype(np.float32)
                                 .astype(np.float64))[0]
        assert_close_abs1(syn.bf16_bits_to_f32(out[t]).astype(np.float64), ref, 2e-2, f"token {t}")
    # the same token alone, and inside a different batch, gives the same bits
    for t in rows[:6]:
        alone, _ = gpu_layer(bi, hidden[t:t + 1], logits[t:t + 1], W1d, W2d)
        assert np.array_equal(alone[0], out[t]), f"token {t}: alone differs from batch of {T}"
    other = np.concatenate([hidden[rows[:6]], syn.to_bf16_bits(syn.normal_rows(9, syn.TID_HIDDEN, 100, HID))])
    other_l = np.concatenate([logits[rows[:6]], syn.normal_rows(9, syn.TID_LOGITS, 100, E)])
    o2, _ = gpu_layer(bi, other, other_l, W1d, W2d)
    for j, t in enumerate(rows[:6]):
        assert np.array_equal(o2[j], out[t]), f"token {t}: changes with co-routed tokens"
    assert bi.device_status() == bi.BI_OK


@pytest.mark.parametrize("T", [1, 7, 64, 512, 8192])
def test_fused_gate_up_silu_equals_unfused(bi, layer_weights, T):
    """bi_grouped_gemm_silu_bf16 gives the bits of bi_grouped_gemm_bf16 followed by
    bi_silu_mul, for every routed row, including partial 256-row expert tiles."""
    _, _, W1d, _ = layer_weights
    tok, exp, off, _ = syn.moe_routing(T, E, TOPK, seed=T)
    X = to_dev_bf16(syn.to_bf16_bits(syn.normal_rows(T, syn.TID_HIDDEN, T, HID))[tok])
    offd = to_dev(off)
    ref = bits_of(bi.silu_mul(bi.grouped_gemm_bf16(X, W1d, offd)))
    got = bits_of(bi.grouped_gemm_silu_bf16(X, W1d, offd))
    assert np.array_equal(got, ref)
    assert bi.device_status() == bi.BI_OK


def test_full_layer_at_the_bench_size_sampled(bi, layer_weights):
    """The size the bench times (T=8192 tokens, the fused gate_up): eight
    sampled tokens against the oracle chain, and each sampled token alone
    gives the same bits."""
    W1, W2, W1d, W2d = layer_weights
    T = 8192
    hidden = syn.to_bf16_bits(syn.normal_rows(8, syn.TID_HIDDEN, T, HID))
    logits = logits_for(T, seed=8)
    out, _ = gpu_layer(bi, hidden, logits, W1d, W2d, fused=True)
    ids, w = oracle.moe_topk_softmax(logits, TOPK)
    for t in [0, 1, 777, 4096, 6000, 8191]:
        ys = []
        for i in range(TOPK):
            e = ids[t, i]
            gu = oracle.bf16_round_array(oracle.gemm_bf16(hidden[t:t + 1], W1[e]))
            act = oracle.bf16_round_array(oracle.silu_mul(gu))
            ys.append(oracle.bf16_round_array(oracle.gemm_bf16(act, W2[e]))[0])
        ref = oracle.moe_combine(np.stack(ys), np.arange(TOPK, dtype=np.int32)[None],
                                 w[t:t + 1].astype(np.float32).astype(np.float64))[0]
        assert_close_abs1(syn.bf16_bits_to_f32(out[t]).astype(np.float64), ref, 2e-2, f"token {t}")
        alone, _ = gpu_layer(bi, hidden[t:t + 1], logits[t:t + 1], W1d, W2d, fused=True)
        assert np.array_equal(alone[0], out[t]), f"token {t}: differs alone"
    assert bi.device_status() == bi.BI_OK


def test_fused_layer_equals_unfused_layer(bi, layer_weights):
    W1, W2, W1d, W2d = layer_weights
    T = 300
    hidden = syn.to_bf16_bits(syn.normal_rows(7, syn.TID_HIDDEN, T, HID))
    logits = logits_for(T, seed=7)
    a, _ = gpu_layer(bi, hidden, logits, W1d, W2d)
    b, _ = gpu_layer(bi, hidden, logits, W1d, W2d, fused=True)
    assert np.array_equal(a, b)


def test_fused_rejects_bad_offsets(bi, layer_weights):
    import torch
    _, _, W1d, _ = layer_weights
    X = torch.zeros((16, HID), dtype=torch.bfloat16, device="cuda")
    off = np.zeros(E + 1, dtype=np.int32)
    off[5:] = 20                         # ends past the 16 rows
    bi.grouped_gemm_silu_bf16(X, W1d, to_dev(off))
    torch.cuda.synchronize()
    assert bi.device_status() == bi.BI_ERR_INVALID_ARG
