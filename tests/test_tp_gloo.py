"""Multi-rank path of the deterministic all-reduce + RMSNorm on CPU (gloo,
world size 2): partials are gathered indexed by rank whatever their arrival
order, and every rank reduces them to the same bits (the fixed-order
reduction vLLM PR #51292 relies on). The reduction itself is computed here by
the oracle; on GPUs it is libbi's bi_rank_sum_rmsnorm."""
import os
import socket

import numpy as np
import pytest

import bi_synth as syn

M, H, EPS = 5, 256, 1e-6


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _partial(rank):
    return syn.to_bf16_bits(syn.normal_rows(100 + rank, syn.TID_X, M, H))


def _worker(rank, world, port, late_rank, q):
    import time
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from invariant_deterministic_bi_gb300 import tp
        x = torch.from_numpy(_partial(rank).view(np.int16)).view(torch.bfloat16)
        if rank == late_rank:
            time.sleep(0.5)
        parts = tp.gather_rank_ordered(x)
        stacked = np.stack([p.view(torch.int16).numpy().view(np.uint16) for p in parts])
        _, res, w, _ = syn.rmsnorm_inputs(M, H, seed=3)
        y, a, h = oracle.rank_sum_rmsnorm(stacked, w, EPS, residual=res)
        q.put((rank, stacked.tobytes(), y.tobytes(), a.tobytes(), h.tobytes()))
    finally:
        dist.destroy_process_group()


def _run(world, late_rank):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, late_rank, q)) for r in range(world)]
    import queue
    import time
    for p in procs:
        p.start()
    out, deadline = [], time.time() + 120
    try:
        while len(out) < world:
            try:
                out.append(q.get(timeout=1))
            except queue.Empty:
                dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                assert not dead, f"a rank exited with {dead}"
                assert time.time() < deadline, "ranks did not report in time"
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.exitcode is None:
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    return sorted(out)


@pytest.mark.parametrize("late_rank", [0, 1])
def test_two_ranks_agree_bit_for_bit(late_rank):
    import oracle
    res = _run(2, late_rank)
    want_parts = np.stack([_partial(0), _partial(1)])
    for rank, parts, y, a, h in res:
        assert parts == want_parts.tobytes(), f"rank {rank}: partials not in rank order"
    assert res[0][2:] == res[1][2:], "ranks disagree"
    _, resid, w, _ = syn.rmsnorm_inputs(M, H, seed=3)
    y, a, h = oracle.rank_sum_rmsnorm(want_parts, w, EPS, residual=resid)
    assert res[0][2] == y.tobytes() and res[0][3] == a.tobytes() and res[0][4] == h.tobytes()


def test_allreduce_rmsnorm_needs_cuda_tensors():
    """The product path has no CPU fallback: CPU tensors are rejected."""
    torch = pytest.importorskip("torch")
    from invariant_deterministic_bi_gb300 import rank_sum_rmsnorm
    x = torch.zeros((2, 8), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        rank_sum_rmsnorm([x], x[0], 1e-6)
