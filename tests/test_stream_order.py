"""Stream order with programmatic dependent launch (every libbi kernel may
start while the previous kernel of the stream finishes, and waits for it
before touching global memory). Chains of calls in which each launch reads
what the previous one wrote, and overwrites what an earlier one read, must
give the same bits back to back, inside a captured CUDA graph, and with the
host synchronising after every call."""
import numpy as np
import pytest

import bi_synth as syn
from util import bits_of, to_dev_bf16

pytestmark = pytest.mark.gpu

M, H, STEPS, EPS = 64, 4096, 16, 1e-6


def inputs():
    x = to_dev_bf16(syn.to_bf16_bits(syn.normal_rows(70, syn.TID_X, M, H)))
    r = to_dev_bf16(syn.to_bf16_bits(syn.normal_rows(71, syn.TID_X, M, H)))
    w = to_dev_bf16(syn.to_bf16_bits(1.0 + 0.1 * syn.normal_rows(72, syn.TID_W, 1, H)[0]))
    W = to_dev_bf16(syn.to_bf16_bits(syn.normal_rows(73, syn.TID_W, H, H, std=0.02)))
    return x, r, w, W


def bf16_chain(bi, x0, r0, w, W, sync: bool):
    """rmsnorm (residual updated in place) -> GEMM, STEPS times; the GEMM writes
    the buffer the rmsnorm before last read (ping-pong)."""
    import torch
    xs = [x0.clone(), torch.empty_like(x0)]
    r = r0.clone()
    y = torch.empty_like(x0)

    def run():
        for i in range(STEPS):
            bi.rmsnorm(xs[i % 2], w, EPS, residual=r, out=y)
            if sync:
                torch.cuda.synchronize()
            bi.gemm_bf16(y, W, Y=xs[(i + 1) % 2])
            if sync:
                torch.cuda.synchronize()
    return xs, r, run


def test_bf16_chain_back_to_back_equals_synchronised(bi):
    import torch
    x, r, w, W = inputs()
    xs_a, r_a, run_a = bf16_chain(bi, x, r, w, W, sync=True)
    run_a()
    xs_b, r_b, run_b = bf16_chain(bi, x, r, w, W, sync=False)
    run_b()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(xs_a[STEPS % 2]), bits_of(xs_b[STEPS % 2]))
    assert np.array_equal(bits_of(r_a), bits_of(r_b))
    assert bi.device_status() == bi.BI_OK


def test_bf16_chain_in_a_graph_equals_synchronised(bi):
    import torch
    x, r, w, W = inputs()
    xs_a, r_a, run_a = bf16_chain(bi, x, r, w, W, sync=True)
    run_a()
    xs_g, r_g, run_g = bf16_chain(bi, x, r, w, W, sync=False)
    run_g()                                       # warm-up outside capture (loads the library)
    torch.cuda.synchronize()
    xs_g[0].copy_(x)
    r_g.copy_(r)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            run_g()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    xs_g[0].copy_(x)                              # capture does not run the work: start from the inputs
    r_g.copy_(r)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(xs_a[STEPS % 2]), bits_of(xs_g[STEPS % 2]))
    assert np.array_equal(bits_of(r_a), bits_of(r_g))


def test_nvfp4_chain_back_to_back_equals_synchronised(bi):
    """rmsnorm -> NVFP4 quantise (into the same Q buffers every step, which the
    previous GEMM read) -> NVFP4 GEMM, STEPS times."""
    import torch
    x, _, w, W = inputs()
    B, B_sf = bi.quantize_nvfp4(W, 1.0)
    torch.cuda.synchronize()

    def chain(sync: bool):
        cur = x.clone()
        y = torch.empty_like(x)
        Q = torch.empty((M, H // 2), dtype=torch.uint8, device="cuda")
        Q_sf = torch.zeros(128 * (H // 16), dtype=torch.uint8, device="cuda")
        for _ in range(STEPS):
            bi.rmsnorm(cur, w, EPS, out=y)
            if sync:
                torch.cuda.synchronize()
            bi.quantize_nvfp4(y, 1.0, Q=Q, Q_sf=Q_sf)
            if sync:
                torch.cuda.synchronize()
            bi.gemm_nvfp4(Q, Q_sf, B, B_sf, 1.0, Y=cur)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return bits_of(cur)

    a = chain(True)
    b = chain(False)
    assert np.isfinite(syn.bf16_bits_to_f32(a)).all()
    assert np.array_equal(a, b)
    assert bi.device_status() == bi.BI_OK


def _capture(fn):
    """Run fn once eagerly (loads the library), then capture it in a CUDA graph
    and replay; returns (eager result, replayed result)."""
    import torch
    eager = fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            out = fn()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    return eager, out, g


def test_attention_and_moe_calls_replay_from_a_graph(bi):
    """Decode attention (with a caller workspace), extend attention and a whole
    MoE layer allocate nothing and synchronise nothing inside the library: captured
    in a CUDA graph and replayed, they give the eager calls' bits."""
    import torch
    g_ = torch.Generator(device="cuda").manual_seed(11)
    Hq, Hkv, D, bs = 32, 8, 128, 16
    lens = torch.tensor([700, 33, 1000], dtype=torch.int32, device="cuda")
    nb = 1000 // bs + 1
    K = torch.randn((3 * nb, bs, Hkv, D), device="cuda", generator=g_).to(torch.bfloat16)
    V = torch.randn((3 * nb, bs, Hkv, D), device="cuda", generator=g_).to(torch.bfloat16)
    table = torch.randperm(3 * nb, device="cuda", generator=g_).to(torch.int32).view(3, nb)
    q = torch.randn((3, Hq, D), device="cuda", generator=g_).to(torch.bfloat16)
    ws = torch.empty(bi.attention_decode_workspace_size(3, Hq, 1000), dtype=torch.uint8, device="cuda")
    dec = lambda: bi.attention_decode(q, K, V, table, lens, 1000, D ** -0.5, workspace=ws, O=torch.empty_like(q))
    a, b, keep1 = _capture(dec)
    assert np.array_equal(bits_of(a), bits_of(b))
    cu = torch.tensor([0, 100, 133, 333], dtype=torch.int32, device="cuda")
    Q = torch.randn((333, Hq, D), device="cuda", generator=g_).to(torch.bfloat16)
    ext = lambda: bi.attention_extend(Q, cu, K, V, table, lens, 1000, 200, D ** -0.5)
    a, b, keep2 = _capture(ext)
    assert np.array_equal(bits_of(a), bits_of(b))
    E, k, T, HID, INTER = 128, 8, 64, 2048, 768
    hidden = torch.randn((T, HID), device="cuda", generator=g_).to(torch.bfloat16)
    logits = torch.randn((T, E), device="cuda", generator=g_)
    W1 = (0.02 * torch.randn((E, 2 * INTER, HID), device="cuda", generator=g_)).to(torch.bfloat16)
    W2 = (0.02 * torch.randn((E, HID, INTER), device="cuda", generator=g_)).to(torch.bfloat16)

    def layer():
        ids, w = bi.moe_topk_softmax(logits, k)
        off, rt, pos = bi.moe_align(ids, E)
        act = bi.grouped_gemm_silu_bf16(bi.moe_gather(hidden, rt), W1, off)
        return bi.moe_combine(bi.grouped_gemm_bf16(act, W2, off), pos, w)
    a, b, keep3 = _capture(layer)
    assert np.array_equal(bits_of(a), bits_of(b))
    assert bi.device_status() == bi.BI_OK


_FIRST_CALLS_IN_A_CAPTURE = r'''
import sys
import torch
sys.path.insert(0, sys.argv[1])
import invariant_deterministic_bi_gb300 as bi

gen = torch.Generator(device="cuda").manual_seed(5)


def bf(*shape, std=1.0):
    return (std * torch.randn(*shape, device="cuda", generator=gen)).to(torch.bfloat16)


x1, r1, w, p0, p1, X = bf(1, 4096), bf(1, 4096), bf(4096), bf(1, 4096), bf(1, 4096), bf(1, 4096)
W = bf(6144, 4096, std=0.02)
Hq, Hkv, L, bs = 32, 8, 4096, 16
K, V = bf(L // bs, bs, Hkv, 128), bf(L // bs, bs, Hkv, 128)
table = torch.arange(L // bs, dtype=torch.int32, device="cuda").view(1, -1)
lens = torch.tensor([L], dtype=torch.int32, device="cuda")
q = bf(1, Hq, 128)
ws = torch.empty(bi.attention_decode_workspace_size(1, Hq, L), dtype=torch.uint8, device="cuda")


def buffers():
    return (r1.clone(), [torch.empty(1, 4096, dtype=torch.bfloat16, device="cuda") for _ in range(2)],
            torch.empty(1, 6144, dtype=torch.bfloat16, device="cuda"), torch.empty_like(q))


def calls(rr, outs, y, o):
    bi.rmsnorm(x1, w, 1e-6, residual=rr, out=outs[0])
    bi.rank_sum_rmsnorm([p0, p1], w, 1e-6, out=outs[1])
    bi.gemm_bf16(X, W, Y=y)
    bi.attention_decode(q, K, V, table, lens, L, 128 ** -0.5, workspace=ws, O=o)


a = buffers()
g = torch.cuda.CUDAGraph()
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
with torch.cuda.stream(side):
    with torch.cuda.graph(g):
        calls(*a)                      # the library's first launches
torch.cuda.current_stream().wait_stream(side)
g.replay()
torch.cuda.synchronize()
b = buffers()
calls(*b)
torch.cuda.synchronize()


def same(u, v):
    return torch.equal(u.view(torch.int16), v.view(torch.int16))


assert same(a[0], b[0]) and all(same(u, v) for u, v in zip(a[1], b[1])) and same(a[2], b[2]) and same(a[3], b[3])
assert bi.device_status() == bi.BI_OK
print("ok")
'''


def test_first_calls_of_a_process_inside_a_capture(bi):
    """A process whose first RMSNorm, rank-sum RMSNorm, GEMM and decode
    attention launches happen inside a CUDA graph capture (the library's
    one-time host queries then run during the capture) replays them with the
    bits of the same calls made eagerly afterwards. A fresh process, so no
    earlier call has done the one-time work."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALLS_IN_A_CAPTURE, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]


_FIRST_MOE_NVFP4_EXTEND_CALLS_IN_A_CAPTURE = r'''
import sys
import torch
sys.path.insert(0, sys.argv[1])
import invariant_deterministic_bi_gb300 as bi

gen = torch.Generator(device="cuda").manual_seed(6)


def bf(*shape, std=1.0):
    return (std * torch.randn(*shape, device="cuda", generator=gen)).to(torch.bfloat16)


T, E, k, H, I = 16, 128, 8, 2048, 768
logits = torch.randn(T, E, device="cuda", generator=gen)
hidden = bf(T, H)
W1, W2 = bf(E, 2 * I, H, std=0.02), bf(E, H, I, std=0.02)
Xq, Wq = bf(16, 256), bf(512, 256)
Hq, Hkv, bs = 32, 8, 16
K, V = bf(64, bs, Hkv, 128), bf(64, bs, Hkv, 128)
table = torch.arange(64, dtype=torch.int32, device="cuda").view(2, 32)
lens = torch.tensor([300, 129], dtype=torch.int32, device="cuda")
cu = torch.tensor([0, 100, 129], dtype=torch.int32, device="cuda")
Qe = bf(129, Hq, 128)


def calls():
    ids, wts = bi.moe_topk_softmax(logits, k)
    off, row_token, pos = bi.moe_align(ids, E)
    xs = bi.moe_gather(hidden, row_token)
    act = bi.grouped_gemm_silu_bf16(xs, W1, off)
    y = bi.grouped_gemm_bf16(act, W2, off)
    out = bi.moe_combine(y, pos, wts)
    qa, sa = bi.quantize_nvfp4(Xq, 1.0)
    qb, sb = bi.quantize_nvfp4(Wq, 1.0)
    yq = bi.gemm_nvfp4(qa, sa, qb, sb, 1.0)
    oe = bi.attention_extend(Qe, cu, K, V, table, lens, 300, 100, 128 ** -0.5)
    return [out, yq, oe]


g = torch.cuda.CUDAGraph()
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
with torch.cuda.stream(side):
    with torch.cuda.graph(g):
        a = calls()                    # the library's first launches
torch.cuda.current_stream().wait_stream(side)
g.replay()
torch.cuda.synchronize()
b = calls()
torch.cuda.synchronize()
assert all(torch.equal(u.view(torch.int16), v.view(torch.int16)) for u, v in zip(a, b))
assert bi.device_status() == bi.BI_OK
print("ok")
'''


def test_first_moe_nvfp4_and_extend_calls_of_a_process_inside_a_capture(bi):
    """The same for a process whose first launches are a whole MoE layer
    (routing, alignment, gather, fused gate_up, down, combine), the NVFP4
    quantiser and GEMM, and extend attention."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_MOE_NVFP4_EXTEND_CALLS_IN_A_CAPTURE, root], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]
