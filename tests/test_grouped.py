"""bi_grouped_gemm_bf16 on the GPU: Qwen3-30B-A3B-shaped MoE expert linears.

128 experts, top-8 routing from seeded router logits, hidden 2048, expert
intermediate 768 (gate_up: K=2048 -> N=1536; down: K=768 -> N=2048). A token's
expert output must not depend on which other tokens share its expert
(batch invariance, vllm-ascend guide; MoE models listed as tested there).
"""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_abs1, bits_of, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
RTOL = 1e-2
E, TOPK, HID, INTER = 128, 8, 2048, 768
LAYERS = {"gate_up": (2 * INTER, HID), "down": (HID, INTER)}


def expert_inputs(T, layer, seed=0):
    N, K = LAYERS[layer]
    tok, exp, off, _ = syn.moe_routing(T, E, TOPK, seed=seed)
    if layer == "gate_up":
        hidden = syn.to_bf16_bits(syn.normal_rows(seed, syn.TID_HIDDEN, T, K))
        X = hidden[tok]
    else:
        X = syn.to_bf16_bits(syn.normal_rows(seed, syn.TID_DOWN_IN, T * TOPK, K))
    W = syn.moe_weights(E, N, K, seed=seed, tensor_id=syn.TID_W1 if layer == "gate_up" else syn.TID_W2)
    return X, W, off, tok, exp


@pytest.fixture(scope="module")
def weights():
    return {layer: syn.moe_weights(E, *LAYERS[layer], seed=0,
                                   tensor_id=syn.TID_W1 if layer == "gate_up" else syn.TID_W2)
            for layer in LAYERS}


@pytest.mark.parametrize("layer", list(LAYERS))
@pytest.mark.parametrize("T", [1, 8, 64, 512, 2048, 8192])
def test_parity_and_token_invariance(bi, weights, layer, T):
    N, K = LAYERS[layer]
    tok, exp, off, _ = syn.moe_routing(T, E, TOPK, seed=0)
    if layer == "gate_up":
        hidden = syn.to_bf16_bits(syn.normal_rows(0, syn.TID_HIDDEN, T, K))
        X = hidden[tok]
    else:
        X = syn.to_bf16_bits(syn.normal_rows(0, syn.TID_DOWN_IN, T * TOPK, K))
    W = weights[layer]
    Wd = to_dev_bf16(W)
    Y = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X), Wd, to_dev(off)))
    rows = sample_rows(T * TOPK, 48, seed=T)
    for r in rows:
        e = int(exp[r])
        ref = oracle.gemm_bf16(X[r:r + 1], W[e])[0]
        assert_close_abs1(syn.bf16_bits_to_f32(Y[r]).astype(np.float64), ref, RTOL, f"{layer} T={T} row {r}")
    # a token routed alone: its rows form groups of one row each
    for t in sorted(set(int(v) for v in tok[rows[:4]])):
        mine = np.nonzero(tok == t)[0]
        counts = np.zeros(E, dtype=np.int64)
        counts[exp[mine]] = 1
        Ya = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X[mine]), Wd, to_dev(syn.offsets_from_counts(counts))))
        assert np.array_equal(Ya, Y[mine]), f"token {t}: expert output changed with co-routed tokens"
    assert bi.device_status() == bi.BI_OK


def test_matches_dense_gemm_per_expert(bi, weights):
    """Each expert's rows equal bi_gemm_bf16 on those rows alone (same K order)."""
    T = 300
    X, W, off, tok, exp = expert_inputs(T, "down")
    Wd = to_dev_bf16(W)
    Y = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X), Wd, to_dev(off)))
    for e in (0, 5, 77, 127):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        Yd = bits_of(bi.gemm_bf16(to_dev_bf16(X[a:b]), Wd[e]))
        assert np.array_equal(Yd, Y[a:b])


def test_empty_experts_ragged_groups_and_exact(bi):
    """Counts with empty experts and groups larger than one M-tile; integer
    inputs make every sum exact, so outputs are bf16(exact sum) bit for bit."""
    counts = [0, 1, 0, 0, 130, 127, 128, 0, 257, 3]
    Ee, N, K = len(counts), 264, 136
    off = syn.offsets_from_counts(counts)
    rows = int(off[-1])
    X = syn.integer_bf16(3, 0, (rows, K))
    W = syn.integer_bf16(3, 1, (Ee, N, K))
    Y = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X), to_dev_bf16(W), to_dev(off)))
    ref = oracle.grouped_gemm_bf16(X, W, off)
    assert np.array_equal(Y, oracle.bf16_round_array(ref))


def test_repeat_and_permuted_groups(bi, weights):
    """8 identical runs give one output; reordering the tokens inside an
    expert's group permutes that group's rows and nothing else."""
    T = 512
    X, W, off, tok, exp = expert_inputs(T, "gate_up")
    Xd, Wd, od = to_dev_bf16(X), to_dev_bf16(W), to_dev(off)
    outs = {bits_of(bi.grouped_gemm_bf16(Xd, Wd, od)).tobytes() for _ in range(8)}
    assert len(outs) == 1
    base = np.frombuffer(outs.pop(), dtype=np.uint16).reshape(X.shape[0], -1)
    perm = np.arange(X.shape[0])
    g = syn.rng(9, 0)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        perm[a:b] = a + g.permutation(b - a)
    Y = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X[perm]), Wd, od))
    assert np.array_equal(Y, base[perm])


@pytest.mark.parametrize("Ee", [1, 33, 100, 1024])
def test_expert_counts_exact(bi, Ee):
    """Expert counts from 1 to the maximum (1024): the device-side tile map
    (a prefix over the experts, split into one block per lane of a warp)
    covers every expert; random group sizes with empty experts and integer
    inputs, so outputs are bf16(exact sum) bit for bit."""
    counts = syn.rng(50 + Ee, 0).integers(0, 6 if Ee > 1 else 300, size=Ee)
    if Ee > 1:
        counts[::7] = 0
    N, K = 264, 136
    off = syn.offsets_from_counts(counts)
    rows = int(off[-1])
    X = syn.integer_bf16(5, 0, (rows, K))
    W = syn.integer_bf16(5, 1, (Ee, N, K))
    Y = bits_of(bi.grouped_gemm_bf16(to_dev_bf16(X), to_dev_bf16(W), to_dev(off)))
    ref = oracle.grouped_gemm_bf16(X, W, off)
    assert np.array_equal(Y, oracle.bf16_round_array(ref))
    assert bi.device_status() == bi.BI_OK
