"""Host-side checks of the seeded input generator (CPU only)."""
import numpy as np

import bi_synth as syn
import oracle


def test_streams_are_prefix_stable():
    a, _ = syn.gemm_inputs(64, 8, 32, seed=0)
    b, _ = syn.gemm_inputs(5, 8, 32, seed=0)
    assert np.array_equal(a[:5], b)


def test_bf16_conversion_matches_torch():
    import torch
    v = syn.normal_rows(0, 99, 64, 64, std=10.0)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(syn.to_bf16_bits(v), ref)


def test_rmsnorm_outlier_rows():
    for M, n in [(1, 0), (3, 0), (128, 1), (4097, 41), (16384, 164)]:
        x, _, _, rows = syn.rmsnorm_inputs(M, 64, seed=0)
        assert len(rows) == n and len(set(rows.tolist())) == n
        if n:
            xf = syn.bf16_bits_to_f32(x)
            big = np.abs(xf[rows]).max(axis=1)
            assert big.min() > 5.0


def test_moe_routing_consistent():
    T, E, k = 257, 128, 8
    tok, exp, off, ids = syn.moe_routing(T, E, k, seed=0)
    assert len(tok) == T * k and off[-1] == T * k and off[0] == 0
    assert np.all(np.diff(off) >= 0)
    for e in range(E):
        seg = slice(off[e], off[e + 1])
        assert np.all(exp[seg] == e)
        assert np.all(np.diff(tok[seg]) > 0)
    for t in range(T):
        assert len(set(ids[t].tolist())) == k


def test_e2m1_encode_rounding():
    v = np.array([0.25, 0.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 7.0, 1.25, 0.0])
    c = syn.e2m1_encode(v)
    got = [oracle.e2m1_value(int(x)) for x in c]
    assert got == [0.0, 1.0, 2.0, 4.0, 4.0, 0.0, -4.0, 6.0, 6.0, 1.0, 0.0]


def test_e2m1_fast_encoder_matches_search():
    g = syn.rng(5, 0)
    v = np.concatenate([g.uniform(-6.5, 6.5, 200000).astype(np.float32),
                        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 0.0, -0.0], np.float32)])
    assert np.array_equal(syn.e2m1_encode(v), syn.e2m1_encode_by_search(v))


def test_e4m3_encode_roundtrip_and_saturation():
    codes = np.arange(0, 127, dtype=np.uint8)
    vals = np.array([oracle.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(syn.e4m3_encode_pos(vals), codes)
    assert syn.e4m3_encode_pos(np.array([1000.0]))[0] == 0x7E


def test_nvfp4_quantise_error_bound():
    d = syn.nvfp4_inputs(8, 16, 256, seed=1)
    a = d["a_f32"].astype(np.float64)
    K = a.shape[1]
    deq = np.zeros_like(a)
    for i in range(a.shape[0]):
        for k in range(K):
            byte = int(d["A"][i, k // 2])
            code = (byte >> 4) if k % 2 else (byte & 15)
            deq[i, k] = oracle.e2m1_value(code) * oracle.e4m3_value(int(d["SA"][i, k // 16])) / float(d["gsa"])
    # per block the e2m1 step is at most 2 (between 4 and 6) in scaled units,
    # so the error is at most one step of the block scale, plus the scale's own rounding.
    blk_amax = np.abs(a).reshape(a.shape[0], K // 16, 16).max(axis=2)
    bound = np.repeat(blk_amax / 6.0 * 1.0 * 1.07, 16, axis=1) + 1e-6
    assert np.all(np.abs(deq - a) <= bound)


def test_swizzle_matches_documented_offsets():
    g = syn.rng(3, 0)
    R, C = 130, 12
    sf = g.integers(0, 127, size=(R, C), dtype=np.uint8)
    il = syn.swizzle_block_scales(sf)
    Cp = 12
    assert il.size == 256 * Cp
    for r in range(R):
        for c in range(C):
            off = ((r // 128) * (Cp // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
            assert il[off] == sf[r, c]
