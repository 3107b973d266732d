"""bi_rank_sum_rmsnorm on one GPU with R emulated ranks (all partials in this
GPU's memory, reduced by one kernel): parity with the oracle, R = 1 equals
bi_rmsnorm bit for bit, rows are independent, repeated runs agree."""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_rel, bits_of, to_dev_bf16

pytestmark = pytest.mark.gpu
EPS = 1e-6


def parts_for(R, M, H, seed=0):
    return np.stack([syn.to_bf16_bits(syn.normal_rows(seed + r, syn.TID_X, M, H)) for r in range(R)])


@pytest.mark.parametrize("R", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 4097])
def test_parity(bi, R, M):
    import torch
    H = 4096
    P = parts_for(R, M, H)
    _, res, w, _ = syn.rmsnorm_inputs(M, H, seed=1)
    pd = [to_dev_bf16(P[r]) for r in range(R)]
    rd = to_dev_bf16(res)
    a_out = torch.empty_like(pd[0])
    out = bi.rank_sum_rmsnorm(pd, to_dev_bf16(w), EPS, residual=rd, sum_out=a_out)
    y, a, h = oracle.rank_sum_rmsnorm(P, w, EPS, residual=res)
    ga = syn.bf16_bits_to_f32(bits_of(a_out)).astype(np.float64)
    # one fp32 rounding of the rank-ordered sum, then bf16: within one bf16 step of the exact rounding
    assert_close_rel(ga, syn.bf16_bits_to_f32(a).astype(np.float64), 2.0 ** -7, 1e-30, "all-reduced rows")
    exact = np.mean(bits_of(a_out) == a)
    assert exact > 0.999, f"only {exact:.4f} of all-reduced values are bit-exact"
    assert_close_rel(syn.bf16_bits_to_f32(bits_of(out)).astype(np.float64), y, 1.6e-2, 1e-6, "out")
    assert bi.device_status() == bi.BI_OK


@pytest.mark.parametrize("R", [3, 5, 16])
@pytest.mark.parametrize("H", [4096, 16384])
def test_rank_order_is_the_stated_one(bi, R, H):
    """The all-reduced row is bf16 of the fp32 sum in rank order 0, 1, ..., R-1
    (each addition rounded to nearest even), bit for bit: numpy float32
    additions in that order give the same bits. Odd R and R = 16 (the
    largest), and a row long enough for the kernel's other loop order."""
    import torch
    M = 37
    P = parts_for(R, M, H, seed=3)
    _, _, w, _ = syn.rmsnorm_inputs(M, H, seed=4)
    pd = [to_dev_bf16(P[r]) for r in range(R)]
    a_out = torch.empty_like(pd[0])
    bi.rank_sum_rmsnorm(pd, to_dev_bf16(w), EPS, sum_out=a_out)
    acc = np.zeros((M, H), dtype=np.float32)
    for r in range(R):
        acc = (acc + syn.bf16_bits_to_f32(P[r])).astype(np.float32)
    assert np.array_equal(bits_of(a_out), syn.to_bf16_bits(acc))
    assert bi.device_status() == bi.BI_OK


def test_rank_order_at_the_bench_size(bi):
    """The size the bench times (R=4 parts of 16384 x 4096, residual in place):
    every all-reduced value bit-exact against float32 additions in rank order,
    the residual update bf16(a + residual) likewise, and the normalised rows
    against the oracle on a sample."""
    import torch
    R, M, H = 4, 16384, 4096
    g = torch.Generator(device="cuda").manual_seed(9)
    pd = [torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16) for _ in range(R)]
    rd = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
    _, _, w, _ = syn.rmsnorm_inputs(1, H, seed=10)
    res0 = bits_of(rd)
    a_out = torch.empty_like(pd[0])
    out = bits_of(bi.rank_sum_rmsnorm(pd, to_dev_bf16(w), EPS, residual=rd, sum_out=a_out))
    assert bi.device_status() == bi.BI_OK
    P = np.stack([bits_of(t) for t in pd])
    acc = np.zeros((M, H), dtype=np.float32)
    for r in range(R):
        acc = (acc + syn.bf16_bits_to_f32(P[r])).astype(np.float32)
    a = syn.to_bf16_bits(acc)
    assert np.array_equal(bits_of(a_out), a)
    h = syn.to_bf16_bits((syn.bf16_bits_to_f32(a) + syn.bf16_bits_to_f32(res0)).astype(np.float32))
    assert np.array_equal(bits_of(rd), h), "residual update"
    rows = [0, 1, 4097, 8191, 16383]
    y, _, _ = oracle.rank_sum_rmsnorm(P[:, rows], w, EPS, residual=res0[rows])
    assert_close_rel(syn.bf16_bits_to_f32(out[rows]).astype(np.float64), y, 1.6e-2, 1e-6, "out")


def test_one_rank_is_rmsnorm(bi):
    M, H = 300, 4096
    x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=2)
    a = bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(x)], to_dev_bf16(w), EPS, residual=to_dev_bf16(res)))
    b = bits_of(bi.rmsnorm(to_dev_bf16(x), to_dev_bf16(w), EPS, residual=to_dev_bf16(res)))
    assert np.array_equal(a, b)


def test_rows_independent_and_repeatable(bi):
    R, M, H = 4, 200, 2048
    P = parts_for(R, M, H, seed=5)
    _, _, w, _ = syn.rmsnorm_inputs(M, H, seed=6)
    wd = to_dev_bf16(w)
    full = bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(P[r]) for r in range(R)], wd, EPS))
    for i in (0, 99, 199):
        one = bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(P[r][i:i + 1]) for r in range(R)], wd, EPS))
        assert np.array_equal(one[0], full[i])
    outs = {bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(P[r]) for r in range(R)], wd, EPS)).tobytes()
            for _ in range(8)}
    assert len(outs) == 1


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("with_res", [False, True])
def test_row_alone_equals_row_in_a_large_batch(bi, R, with_res):
    """A row reduced alone (M = 1) and among M = 4097 rows gives the same bits,
    output and updated residual: the two sizes launch different forms of the
    kernel (the row's residual and weight vectors loaded before or after the
    rank sum; two or four ranks' loads in flight), which compute the same
    operations in the same order."""
    M, H = 4097, 4096
    P = parts_for(R, M, H, seed=7)
    _, res, w, _ = syn.rmsnorm_inputs(M, H, seed=8)
    wd = to_dev_bf16(w)
    rd = to_dev_bf16(res) if with_res else None
    full = bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(P[r]) for r in range(R)], wd, EPS, residual=rd))
    for i in (0, 2048, 4096):
        r1 = to_dev_bf16(res[i:i + 1]) if with_res else None
        one = bits_of(bi.rank_sum_rmsnorm([to_dev_bf16(P[r][i:i + 1]) for r in range(R)], wd, EPS, residual=r1))
        assert np.array_equal(one[0], full[i]), f"row {i}"
        if with_res:
            assert np.array_equal(bits_of(r1)[0], bits_of(rd)[i]), f"residual row {i}"
    assert bi.device_status() == bi.BI_OK
