"""bi_rmsnorm on the GPU: parity with the fp64 oracle, exact residual, invariance."""
import numpy as np
import pytest

import bi_synth as syn
import oracle
from util import assert_close_rel, bits_of, sample_rows, to_dev_bf16

pytestmark = pytest.mark.gpu
RTOL, ATOL = 8e-3, 1e-6
EPS = 1e-6


def _run(bi, x, w, res=None):
    import torch
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    rd = to_dev_bf16(res) if res is not None else None
    out = bi.rmsnorm(xd, wd, EPS, residual=rd)
    torch.cuda.synchronize()
    return bits_of(out), (bits_of(rd) if rd is not None else None)


@pytest.mark.parametrize("M", [1, 3, 128, 4097, 16384])
@pytest.mark.parametrize("with_res", [False, True])
def test_parity_and_invariance(bi, M, with_res):
    H = 4096
    x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=0)
    r = res if with_res else None
    out, h = _run(bi, x, w, r)
    rows = sample_rows(M, 64, seed=M) if M > 256 else np.arange(M)
    ref, href = oracle.rmsnorm(x[rows], w, EPS, residual=r[rows] if with_res else None)
    assert_close_rel(syn.bf16_bits_to_f32(out[rows]).astype(np.float64), ref, RTOL, ATOL, f"M={M}")
    if with_res:
        assert np.array_equal(h[rows], href), "residual out must be bf16(x + residual) exactly"
    for i in rows[:8]:
        o1, h1 = _run(bi, x[i:i + 1], w, r[i:i + 1] if with_res else None)
        assert np.array_equal(o1[0], out[i]), f"row {i} differs between M={M} and M=1"


@pytest.mark.parametrize("H", [8, 264, 1024, 8192, 12288])
def test_other_hidden_sizes(bi, H):
    M = 37
    x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=H, outlier_frac=0.1)
    out, h = _run(bi, x, w, res)
    ref, href = oracle.rmsnorm(x, w, EPS, residual=res)
    assert_close_rel(syn.bf16_bits_to_f32(out).astype(np.float64), ref, RTOL, ATOL, f"H={H}")
    assert np.array_equal(h, href)
    out2, _ = _run(bi, x, w)
    ref2, _ = oracle.rmsnorm(x, w, EPS)
    assert_close_rel(syn.bf16_bits_to_f32(out2).astype(np.float64), ref2, RTOL, ATOL, f"H={H} no residual")


def test_permutation_repeat_and_in_place(bi):
    import torch
    M, H = 300, 4096
    x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=5)
    base, _ = _run(bi, x, w, res)
    perm = syn.permutation(5, M)
    p, _ = _run(bi, x[perm], w, res[perm])
    assert np.array_equal(p, base[perm])
    outs = {_run(bi, x, w, res)[0].tobytes() for _ in range(8)}
    assert len(outs) == 1
    xd = to_dev_bf16(x)
    bi.rmsnorm(xd, to_dev_bf16(w), EPS, residual=to_dev_bf16(res), out=xd)   # out aliases x
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(xd), base)


def test_special_rows(bi):
    """Zero row -> 0; constant row -> c / sqrt(c^2 + eps) * w (closed form)."""
    H = 4096
    x = np.zeros((3, H), dtype=np.float32)
    x[1] = 1.0
    x[2] = -3.5
    w = np.ones(H, dtype=np.float32)
    out, _ = _run(bi, syn.to_bf16_bits(x), syn.to_bf16_bits(w))
    y = syn.bf16_bits_to_f32(out)
    assert np.all(y[0] == 0)
    assert np.all(y[1] == 1.0)
    assert np.all(y[2] == -1.0)


@pytest.mark.parametrize("H", [264, 8192])
def test_row_alone_equals_row_in_a_large_batch_other_widths(bi, H):
    """A row normalised alone (M = 1) and among M = 4097 rows gives the same
    bits, output and updated residual, at a ragged width (33 vectors of 8)
    and a long one (8 vectors a thread): with the residual the two sizes run
    the kernel's two forms (weight vectors loaded with the row or after the
    reduction), which compute the same operations."""
    M = 4097
    x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=H + 1)
    out, h = _run(bi, x, w, res)
    for i in (0, 2048, 4096):
        o1, h1 = _run(bi, x[i:i + 1], w, res[i:i + 1])
        assert np.array_equal(o1[0], out[i]), f"row {i}"
        assert np.array_equal(h1[0], h[i]), f"residual row {i}"
