"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: brute force
in exact rational arithmetic on small integer or dyadic inputs, closed forms,
hand-worked fixtures under tests/golden/, the storage-format definitions, or an
independent library routine. They are chosen so that a dropped term, a wrong
sign or index, a transposed operand or a misplaced eps fails at least one.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import bi_synth as syn
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s: str):
    return None if s == "NaN" else Fraction(s)


def _bf16_frac(bits: int) -> Fraction:
    return Fraction(float(syn.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0]))


# ------------------------------------------------------------------ formats

def test_format_tables_match_golden():
    n = 0
    with open(os.path.join(GOLDEN, "formats.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            fmt, code, val = line.split()
            code = int(code, 16)
            want = _frac(val)
            got = oracle.e2m1_value(code) if fmt == "e2m1" else oracle.e4m3_value(code)
            if want is None:
                assert math.isnan(got)
            else:
                assert Fraction(got) == want, (fmt, hex(code), got, want)
            n += 1
    assert n >= 30


def test_e4m3_matches_torch_float8():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e2m1_structure():
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals[:8] == sorted(vals[:8])                   # positive codes increase
    assert all(vals[c + 8] == -vals[c] for c in range(8))  # bit 3 is the sign
    assert max(vals) == 6.0


def test_bf16_round_golden():
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, bits = line.split()
            assert oracle.bf16_round(float(Fraction(v))) == int(bits, 16), line


def test_bf16_round_array_matches_scalar():
    v = np.array([1.0, 257 / 256, 259 / 256, -3.0, 1 / 3, 65408.0, 0.0, 1e-40, -2.5e38])
    assert [int(b) for b in oracle.bf16_round_array(v)] == [oracle.bf16_round(x) for x in v]


def test_bf16_round_exhaustive_against_neighbours():
    """Round-trip every positive finite bf16 and check midpoints between
    neighbours go to the even pattern (ties-to-even, by construction)."""
    bits = np.arange(0x0001, 0x7F80, 37, dtype=np.uint16)
    for b in bits:
        v = oracle.bf16_value(int(b))
        assert oracle.bf16_round(v) == b
        nxt = oracle.bf16_value(int(b) + 1)
        mid = (Fraction(v) + Fraction(nxt)) / 2
        want = b if b % 2 == 0 else b + 1
        assert oracle.bf16_round(float(mid)) == want


# -------------------------------------------------------------------- GEMM

def _brute_gemm(X_bits, W_bits):
    X = [[_bf16_frac(int(v)) for v in row] for row in X_bits]
    W = [[_bf16_frac(int(v)) for v in row] for row in W_bits]
    return [[sum(x * w for x, w in zip(xr, wr)) for wr in W] for xr in X]


@pytest.mark.parametrize("M,N,K", [(5, 7, 64), (3, 11, 256), (1, 16, 48)])
def test_gemm_exact_vs_bruteforce(M, N, K):
    X = syn.integer_bf16(1, 0, (M, K))
    W = syn.integer_bf16(1, 1, (N, K))
    Y = oracle.gemm_bf16(X, W)
    ref = _brute_gemm(X, W)
    for i in range(M):
        for j in range(N):
            assert Fraction(Y[i, j]) == ref[i][j]


def test_gemm_identity_and_onehot():
    K = 32
    X = syn.integer_bf16(2, 0, (6, K))
    eye = syn.to_bf16_bits(np.eye(K, dtype=np.float32))
    assert np.array_equal(oracle.gemm_bf16(X, eye), syn.bf16_bits_to_f32(X).astype(np.float64))
    W = syn.integer_bf16(2, 1, (9, K))
    for k in (0, 5, K - 1):
        onehot = np.zeros((1, K), dtype=np.float32)
        onehot[0, k] = 1.0
        Y = oracle.gemm_bf16(syn.to_bf16_bits(onehot), W)
        assert np.array_equal(Y[0], syn.bf16_bits_to_f32(W[:, k]).astype(np.float64))


def test_gemm_close_to_numpy_fp64():
    X, W = syn.gemm_inputs(17, 40, 256, seed=3)
    Y = oracle.gemm_bf16(X, W)
    ref = syn.bf16_bits_to_f32(X).astype(np.float64) @ syn.bf16_bits_to_f32(W).astype(np.float64).T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_rows_independent_of_batch():
    """Oracle-level invariance: row i alone equals row i of the batch."""
    X, W = syn.gemm_inputs(9, 24, 128, seed=4)
    full = oracle.gemm_bf16(X, W)
    for i in range(9):
        assert np.array_equal(oracle.gemm_bf16(X[i:i + 1], W)[0], full[i])


def test_grouped_vs_bruteforce():
    E, N, K = 5, 6, 32
    counts = [3, 0, 1, 4, 0]
    off = syn.offsets_from_counts(counts)
    X = syn.integer_bf16(5, 0, (int(off[-1]), K))
    W = syn.integer_bf16(5, 1, (E, N, K))
    Y = oracle.grouped_gemm_bf16(X, W, off)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            ref = _brute_gemm(X[r:r + 1], W[e])[0]
            assert [Fraction(v) for v in Y[r]] == ref


# ------------------------------------------------------------------- NVFP4

def _brute_nvfp4(A, SA, B, SB, alpha):
    def deq(q, s, i, k):
        byte = int(q[i, k // 2])
        code = (byte >> 4) if k % 2 else (byte & 15)
        return Fraction(oracle.e2m1_value(code)) * Fraction(oracle.e4m3_value(int(s[i, k // 16])))
    M, N, K = A.shape[0], B.shape[0], A.shape[1] * 2
    return [[Fraction(alpha) * sum(deq(A, SA, i, k) * deq(B, SB, j, k) for k in range(K))
             for j in range(N)] for i in range(M)]


def test_nvfp4_exact_vs_bruteforce():
    g = syn.rng(7, 0)
    M, N, K = 3, 5, 64
    A = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    SA = g.integers(0x30, 0x41, size=(M, K // 16), dtype=np.uint8)   # 0.5 .. 2
    SB = g.integers(0x30, 0x41, size=(N, K // 16), dtype=np.uint8)
    alpha = 0.25
    Y = oracle.gemm_nvfp4(A, SA, B, SB, alpha)
    ref = _brute_nvfp4(A, SA, B, SB, alpha)
    for i in range(M):
        for j in range(N):
            assert Fraction(Y[i, j]) == ref[i][j]


def test_nvfp4_nibble_order_and_scale_index():
    """One nonzero element at an odd k in block 2: only the high nibble of
    byte k/2 and scale k/16 may contribute."""
    K = 64
    A = np.zeros((1, K // 2), dtype=np.uint8)
    B = np.zeros((1, K // 2), dtype=np.uint8)
    k = 37                               # odd -> high nibble; block 37//16 = 2
    A[0, k // 2] = 0x2 << 4              # +1.0 in the high nibble
    B[0, k // 2] = (0x7 << 4) | 0x5      # +6.0 high, +3.0 low (k = 36)
    SA = np.full((1, 4), 0x38, dtype=np.uint8)
    SB = np.full((1, 4), 0x38, dtype=np.uint8)
    SA[0, 2] = 0x40                      # 2.0 for block 2
    SB[0, 1] = 0x48                      # a wrong block index would pick up 4.0
    Y = oracle.gemm_nvfp4(A, SA, B, SB, 1.0)
    assert Y[0, 0] == 1.0 * 2.0 * 6.0


def test_nvfp4_unit_scales_integer_case():
    """Unit scales, alpha 1: the result is a plain dot product of e2m1 values."""
    g = syn.rng(8, 0)
    codes_a = g.integers(0, 16, size=(2, 128))
    codes_b = g.integers(0, 16, size=(4, 128))
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    one = lambda r: np.full((r, 8), 0x38, dtype=np.uint8)
    Y = oracle.gemm_nvfp4(pack(codes_a), one(2), pack(codes_b), one(4), 1.0)
    tab = syn._E2M1
    val = lambda c: np.where(c >= 8, -tab[c & 7], tab[c & 7])
    assert np.array_equal(Y, val(codes_a) @ val(codes_b).T)


# ----------------------------------------------------------- quantiser

def test_quantize_golden_blocks():
    n = 0
    with open(os.path.join(GOLDEN, "nvfp4_quant_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            case, gs, xs, sc, qb = line.split()
            x = np.array([float(v) for v in xs.split(",")], dtype=np.float32)[None]
            Xb = syn.to_bf16_bits(x)
            assert np.array_equal(syn.bf16_bits_to_f32(Xb), x), "fixture values must be exact in bf16"
            Q, S = oracle.quantize_nvfp4(Xb, float(gs))
            assert int(S[0, 0]) == int(sc, 16), (case, hex(int(S[0, 0])))
            assert [int(b) for b in Q[0]] == [int(v, 16) for v in qb.split(",")], (case, [hex(b) for b in Q[0]])
            n += 1
    assert n == 7


def test_e4m3_encoder_roundtrip_ties_saturation():
    for c in range(0x7F):
        v = oracle.e4m3_value(c)
        assert oracle.e4m3_encode(v) == c
        if c < 0x7E:
            mid = (Fraction(v) + Fraction(oracle.e4m3_value(c + 1))) / 2
            assert oracle.e4m3_encode(float(mid)) == (c if c % 2 == 0 else c + 1)
    for v in (448.0, 460.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E


def test_e4m3_encoder_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    g = syn.rng(31, 0)
    v = np.exp(g.uniform(np.log(2.0 ** -10), np.log(440.0), 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e2m1_encoder_ties_and_clamp():
    cases = {0.0: 0, 0.24: 0, 0.25: 0, 0.26: 1, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6,
             5.0: 6, 5.01: 7, 6.0: 7, 9.0: 7, -0.25: 0, -0.3: 9, -5.0: 14}
    for v, c in cases.items():
        assert oracle.e2m1_encode(v) == c, v


def test_quantize_agrees_with_generator_quantiser():
    """Two independent implementations of the same reading (this oracle and
    the input generator) agree code for code on random data."""
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(syn.normal_rows(4, 0, 64, 512)))
    x[3] *= 40.0
    x[5, :16] = 0.0
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(x))
    gs = syn.nvfp4_global_scale(x)
    Q, S = oracle.quantize_nvfp4(syn.to_bf16_bits(x), gs)
    Qg, Sg = syn.nvfp4_quantize(x, gs)
    assert np.array_equal(S, Sg) and np.array_equal(Q, Qg)


def test_quantize_dequant_error_bound():
    x = syn.bf16_bits_to_f32(syn.to_bf16_bits(syn.normal_rows(5, 0, 16, 256)))
    gs = syn.nvfp4_global_scale(x)
    Q, S = oracle.quantize_nvfp4(syn.to_bf16_bits(x), gs)
    for i in range(16):
        for k in range(256):
            code = (int(Q[i, k // 2]) >> 4) if k % 2 else (int(Q[i, k // 2]) & 15)
            s = oracle.e4m3_value(int(S[i, k // 16]))
            deq = oracle.e2m1_value(code) * s / float(gs)
            amax = np.abs(x[i, (k // 16) * 16:(k // 16) * 16 + 16]).max()
            # half the largest e2m1 step (1.0 of 6 units) times the block scale, plus scale rounding
            assert abs(deq - x[i, k]) <= amax / 6 * 1.07 + 1e-7


# ------------------------------------------------------------- MoE layer

def test_topk_softmax_hand_worked():
    """logits [1, 3, 3, 0], k = 2: experts 1 and 2 tie, the lower index comes
    first; renormalised weights are 1/2 each; raw softmax weights are
    e^3 / (e + 2 e^3 + 1)."""
    l = np.array([[1.0, 3.0, 3.0, 0.0]], dtype=np.float32)
    ids, w = oracle.moe_topk_softmax(l, 2, renormalize=True)
    assert ids.tolist() == [[1, 2]] and np.allclose(w, 0.5, rtol=0, atol=1e-15)
    ids, w = oracle.moe_topk_softmax(l, 2, renormalize=False)
    p = math.exp(3) / (math.e + 2 * math.exp(3) + 1)
    assert np.allclose(w, p, rtol=1e-14)


def test_topk_softmax_vs_numpy_scipy():
    scipy = pytest.importorskip("scipy.special")
    l = syn.normal_rows(6, 0, 50, 128)
    l[3, 10] = l[3, 20] = l[3].max() + 1     # an exact tie at the top
    ids, w = oracle.moe_topk_softmax(l, 8, renormalize=False)
    ref_ids = np.argsort(-l, axis=1, kind="stable")[:, :8]
    assert np.array_equal(ids, ref_ids)
    p = scipy.softmax(l.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, ref_ids, axis=1), rtol=1e-12)
    ids2, w2 = oracle.moe_topk_softmax(l, 8, renormalize=True)
    assert np.array_equal(ids2, ids) and np.allclose(w2.sum(axis=1), 1.0, rtol=1e-14)


def test_align_matches_stable_sort_and_inverts():
    T, E, k = 300, 128, 8
    tok, exp, off, ids = syn.moe_routing(T, E, k, seed=7)
    o_off, o_row_token, o_pos = oracle.moe_align(ids, E)
    assert np.array_equal(o_off, off) and np.array_equal(o_row_token, tok)
    flat = o_pos.reshape(-1)
    assert sorted(flat.tolist()) == list(range(T * k))       # a bijection
    for t in range(T):
        for i in range(k):
            r = o_pos[t, i]
            assert o_row_token[r] == t and off[ids[t, i]] <= r < off[ids[t, i] + 1]


def test_silu_mul_closed_forms():
    scipy = pytest.importorskip("scipy.special")
    g = np.array([[0.0, 1.0, -2.0, 10.0, -30.0, 0.5, 3.0, -0.25]], dtype=np.float32)
    u = np.array([[5.0, 2.0, 1.0, 0.5, 4.0, -1.0, 0.0, 8.0]], dtype=np.float32)
    gu = syn.to_bf16_bits(np.concatenate([g, u], axis=1))
    act = oracle.silu_mul(gu)
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    assert act[0, 0] == 0.0 and act[0, 6] == 0.0
    assert np.allclose(act, gd * scipy.expit(gd) * ud, rtol=1e-14, atol=0)


def test_combine_bruteforce():
    Y = syn.integer_bf16(8, 0, (12, 16), lo=-4, hi=4)
    pos = np.array([[3, 0, 7], [11, 2, 2], [5, 6, 1]], dtype=np.int32)
    w = np.array([[0.5, 0.25, 0.125], [1.0, -0.5, 0.5], [0.0, 2.0, 0.75]])
    out = oracle.moe_combine(Y, pos, w)
    Yf = syn.bf16_bits_to_f32(Y).astype(np.float64)
    for t in range(3):
        ref = sum(Fraction(w[t, i]) * np.array([Fraction(v) for v in Yf[pos[t, i]]]) for i in range(3))
        assert [Fraction(v) for v in out[t]] == list(ref)


# ------------------------------------------------------------ attention

def _paged(B, L, Hkv, D, bs, seed, lens=None):
    """Random contiguous K/V per sequence, stored in shuffled physical blocks."""
    lens = np.full(B, L, dtype=np.int32) if lens is None else np.asarray(lens, dtype=np.int32)
    nb = -(-lens.max() // bs)
    blocks = B * nb
    K = syn.to_bf16_bits(syn.normal_rows(seed, 0, blocks * bs, Hkv * D)).reshape(blocks, bs, Hkv, D)
    V = syn.to_bf16_bits(syn.normal_rows(seed, 1, blocks * bs, Hkv * D)).reshape(blocks, bs, Hkv, D)
    table = syn.rng(seed, 2).permutation(blocks).astype(np.int32).reshape(B, nb)
    return K, V, table, lens


def _dense(K, V, table, lens, b):
    bs = K.shape[1]
    L = lens[b]
    idx = [(table[b, j // bs], j % bs) for j in range(L)]
    return (np.stack([K[p, o] for p, o in idx]), np.stack([V[p, o] for p, o in idx]))   # [L, Hkv, D]


def test_attention_single_token_and_uniform_keys():
    B, Hq, Hkv, D, bs = 1, 4, 2, 16, 4
    Q = syn.to_bf16_bits(syn.normal_rows(1, 0, B * Hq, D)).reshape(B, Hq, D)
    K, V, table, lens = _paged(B, 1, Hkv, D, bs, seed=2)
    O = oracle.attention_decode(Q, K, V, table, lens, 0.125)
    k0, v0 = _dense(K, V, table, lens, 0)
    for h in range(Hq):
        assert np.array_equal(O[0, h], syn.bf16_bits_to_f32(v0[0, h // 2]).astype(np.float64))
    # identical keys: uniform weights, output = mean of the values (integers, L = 4: exact)
    K4 = np.zeros((1, 4, Hkv, D), dtype=np.uint16) + syn.to_bf16_bits(np.float32(0.5))
    V4 = syn.integer_bf16(3, 0, (1, 4, Hkv, D))
    O4 = oracle.attention_decode(Q, K4, V4, np.zeros((1, 1), np.int32), np.array([4], np.int32), 1.0)
    for h in range(Hq):
        assert np.array_equal(O4[0, h], syn.bf16_bits_to_f32(V4[0, :, h // 2]).astype(np.float64).mean(axis=0))


def test_attention_matches_dense_numpy():
    scipy = pytest.importorskip("scipy.special")
    B, Hq, Hkv, D, bs = 3, 8, 2, 64, 16
    lens = [37, 1, 100]
    Q = syn.to_bf16_bits(syn.normal_rows(4, 0, B * Hq, D)).reshape(B, Hq, D)
    K, V, table, lens = _paged(B, 0, Hkv, D, bs, seed=5, lens=lens)
    scale = 1 / np.sqrt(D)
    O = oracle.attention_decode(Q, K, V, table, lens, scale)
    for b in range(B):
        kd, vd = _dense(K, V, table, lens, b)
        kf = syn.bf16_bits_to_f32(kd).astype(np.float64)
        vf = syn.bf16_bits_to_f32(vd).astype(np.float64)
        for h in range(Hq):
            q = syn.bf16_bits_to_f32(Q[b, h]).astype(np.float64)
            p = scipy.softmax(kf[:, h // 4] @ q * scale)
            assert np.allclose(O[b, h], p @ vf[:, h // 4], rtol=1e-12, atol=1e-14)


def test_attention_block_placement_does_not_matter():
    B, Hq, Hkv, D, bs = 2, 4, 1, 32, 8
    Q = syn.to_bf16_bits(syn.normal_rows(6, 0, B * Hq, D)).reshape(B, Hq, D)
    K, V, table, lens = _paged(B, 50, Hkv, D, bs, seed=7)
    O = oracle.attention_decode(Q, K, V, table, lens, 0.2)
    perm = syn.rng(8, 0).permutation(K.shape[0])
    inv = np.argsort(perm)
    O2 = oracle.attention_decode(Q, K[perm], V[perm], inv[table].astype(np.int32), lens, 0.2)
    assert np.array_equal(O, O2)


def _extend_inputs(lens, qlens, Hq, Hkv, D, bs, seed):
    B = len(lens)
    K, V, table, lens = _paged(B, 0, Hkv, D, bs, seed=seed, lens=lens)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    Q = syn.to_bf16_bits(syn.normal_rows(seed + 1, 0, int(cu[-1]) * Hq, D)).reshape(int(cu[-1]), Hq, D)
    return Q, cu, K, V, table, lens


def test_attention_extend_matches_causal_numpy():
    """Each new token attends to the tokens up to its own position (a causal
    mask over the cached sequence), checked against scipy's softmax."""
    scipy = pytest.importorskip("scipy.special")
    Hq, Hkv, D, bs = 4, 2, 32, 8
    lens, qlens = [19, 6, 40], [5, 6, 1]
    Q, cu, K, V, table, lens = _extend_inputs(lens, qlens, Hq, Hkv, D, bs, seed=11)
    scale = 1 / np.sqrt(D)
    O = oracle.attention_extend(Q, cu, K, V, table, lens, scale)
    for b in range(len(lens)):
        kd, vd = _dense(K, V, table, lens, b)
        kf, vf = (syn.bf16_bits_to_f32(a).astype(np.float64) for a in (kd, vd))
        for i in range(qlens[b]):
            t, pos = cu[b] + i, lens[b] - qlens[b] + i
            for h in range(Hq):
                q = syn.bf16_bits_to_f32(Q[t, h]).astype(np.float64)
                pr = scipy.softmax(kf[:pos + 1, h // 2] @ q * scale)
                assert np.allclose(O[t, h], pr @ vf[:pos + 1, h // 2], rtol=1e-12, atol=1e-14)


def test_attention_extend_of_one_token_is_decode():
    """One new token per sequence: extend is decode attention over the whole cache."""
    Hq, Hkv, D, bs = 8, 2, 64, 16
    lens = [37, 1, 130]
    Q, cu, K, V, table, lens = _extend_inputs(lens, [1, 1, 1], Hq, Hkv, D, bs, seed=13)
    O = oracle.attention_extend(Q, cu, K, V, table, lens, 0.1)
    assert np.array_equal(O, oracle.attention_decode(Q, K, V, table, lens, 0.1))


def test_attention_extend_is_causal():
    """Changing the keys and values after a token's position leaves its output alone."""
    Hq, Hkv, D, bs = 2, 1, 16, 4
    Q, cu, K, V, table, lens = _extend_inputs([12], [12], Hq, Hkv, D, bs, seed=17)
    O = oracle.attention_extend(Q, cu, K, V, table, lens, 0.3)
    K2, V2 = K.copy(), V.copy()
    late = table[0, 2]                       # block of positions 8 .. 11
    K2[late] = syn.to_bf16_bits(syn.normal_rows(18, 0, bs, Hkv * D)).reshape(bs, Hkv, D)
    V2[late] = syn.to_bf16_bits(syn.normal_rows(19, 0, bs, Hkv * D)).reshape(bs, Hkv, D)
    O2 = oracle.attention_extend(Q, cu, K2, V2, table, lens, 0.3)
    assert np.array_equal(O[:8], O2[:8]) and not np.array_equal(O[8:], O2[8:])


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_golden_cases():
    with open(os.path.join(GOLDEN, "rmsnorm_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            _, eps, h, w, y = line.split()
            h = np.array([float(v) for v in h.split(",")], dtype=np.float32)[None]
            w = np.array([float(v) for v in w.split(",")], dtype=np.float32)
            want = np.array([float(v) for v in y.split(",")])
            got, _ = oracle.rmsnorm(syn.to_bf16_bits(h), syn.to_bf16_bits(w), float(eps))
            assert np.allclose(got[0], want, rtol=1e-13, atol=1e-15), (line, got)


@pytest.mark.parametrize("c", [1.0, 0.001, 37.5, -2.0])
def test_rmsnorm_constant_row_closed_form(c):
    H, eps = 64, 1e-6
    x = syn.to_bf16_bits(np.full((1, H), c, dtype=np.float32))
    w = syn.to_bf16_bits(np.linspace(0.5, 1.5, H).astype(np.float32))
    cb = oracle.bf16_value(int(x[0, 0]))
    y, _ = oracle.rmsnorm(x, w, eps)
    want = cb / math.sqrt(cb * cb + eps) * syn.bf16_bits_to_f32(w).astype(np.float64)
    assert np.allclose(y[0], want, rtol=1e-14, atol=0)


def test_rmsnorm_scale_invariance():
    x, _, w, _ = syn.rmsnorm_inputs(4, 256, seed=9, outlier_frac=0)
    y1, _ = oracle.rmsnorm(x, w, 0.0)
    x2 = syn.to_bf16_bits(syn.bf16_bits_to_f32(x) * np.float32(64.0))   # exact power-of-two scaling
    y2, _ = oracle.rmsnorm(x2, w, 0.0)
    assert np.allclose(y1, y2, rtol=1e-14, atol=1e-15)


def test_rmsnorm_residual_is_rounded_sum():
    x = syn.to_bf16_bits(np.array([[1.0, 1.0, 2.0, -3.0]], dtype=np.float32))
    r = syn.to_bf16_bits(np.array([[2.0 ** -8, 3 * 2.0 ** -8, 2.0 ** -7, 0.5]], dtype=np.float32))
    w = syn.to_bf16_bits(np.ones(4, dtype=np.float32))
    y, h = oracle.rmsnorm(x, w, 1e-6, residual=r)
    assert list(h[0]) == [0x3F80, 0x3F82, 0x4000, 0xC020]   # ties to even; 2+2^-7 -> 2; -2.5
    hv = np.array([1.0, 1.0 + 2 ** -6, 2.0, -2.5])
    want = hv / math.sqrt(np.mean(hv ** 2) + 1e-6)
    assert np.allclose(y[0], want, rtol=1e-14)


def test_rank_sum_rmsnorm_reduces_to_rmsnorm_and_sums_exactly():
    x, res, w, _ = syn.rmsnorm_inputs(6, 256, seed=11)
    # one rank: exactly RMSNorm
    y1, a1, h1 = oracle.rank_sum_rmsnorm(x[None], w, 1e-6, residual=res)
    y0, h0 = oracle.rmsnorm(x, w, 1e-6, residual=res)
    assert np.array_equal(a1, x) and np.array_equal(h1, h0) and np.array_equal(y1, y0)
    # x and -x cancel exactly: the all-reduced rows are zero, the output is zero
    neg = x ^ np.uint16(0x8000)
    y2, a2, _ = oracle.rank_sum_rmsnorm(np.stack([x, neg]), w, 1e-6)
    assert np.all(syn.bf16_bits_to_f32(a2) == 0) and np.all(y2 == 0)
    # small integers: the all-reduced value is the integer sum (exact in bf16 below 256)
    parts = syn.integer_bf16(3, 0, (4, 5, 64), lo=-30, hi=30)
    _, a3, _ = oracle.rank_sum_rmsnorm(parts, w[:64], 1e-6)
    assert np.array_equal(syn.bf16_bits_to_f32(a3), syn.bf16_bits_to_f32(parts).sum(axis=0))
    # the all-reduce rounds once: 1 + 2^-8 + 2^-8 = 1 + 2^-7 exactly (two partial
    # roundings would give 1.0)
    one = syn.to_bf16_bits(np.array([[[1.0] * 8]], dtype=np.float32))
    tiny = syn.to_bf16_bits(np.array([[[2.0 ** -8] * 8]], dtype=np.float32))
    _, a4, _ = oracle.rank_sum_rmsnorm(np.concatenate([one, tiny, tiny]), w[:8], 1e-6)
    assert np.all(a4 == 0x3F81)


def test_rmsnorm_rows_independent():
    x, res, w, _ = syn.rmsnorm_inputs(7, 128, seed=10)
    full, hfull = oracle.rmsnorm(x, w, 1e-6, residual=res)
    for i in range(7):
        yi, hi = oracle.rmsnorm(x[i:i + 1], w, 1e-6, residual=res[i:i + 1])
        assert np.array_equal(yi[0], full[i]) and np.array_equal(hi[0], hfull[i])
