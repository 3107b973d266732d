"""Benchmark of the batch-invariant linear layer and RMSNorm (libbi) on GB300.

Headline step (one pass of the hot path over one batch, Qwen3-8B-shaped
decoder-layer linears at M = 8192 tokens, bf16, synthetic N(0,1) activations and
N(0, 0.02^2) weights):
    RMSNorm + residual add [M, 4096]   -> qkv     Y = X W^T  K=4096  N=6144
    RMSNorm + residual add [M, 4096]   -> gate_up Y = X W^T  K=4096  N=24576
    down   Y = X W^T  K=12288 N=4096   (X = first 12288 columns of gate_up's output)
value = GEMM FLOPs of the step / device time of the step (TFLOP/s); the step's
working set (> 1 GB of weights and activations) is far larger than the 129 MB
L2, so back-to-back steps do not hit in L2.

Also reported on the same line: the roofline of the dominant kernel
(bi_gemm_bf16), an end-to-end number through host buffers, the fp64 CPU oracle
timed on a bounded sample, and per-row measurements (M sweep vs cuBLAS,
RMSNorm GB/s vs torch, MoE grouped GEMM, NVFP4 GEMM when present).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 (torchrun) every rank runs an independent replica (no collectives).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_STEP = 8192
H = 4096
EPS = 1e-6
LAYERS = {"qkv": (6144, 4096), "gate_up": (24576, 4096), "down": (4096, 12288)}
M_SWEEP = [1, 7, 64, 513, 4096, 8192]
RMS_SWEEP = [1, 3, 128, 4097, 16384]
METRIC = "batch-invariant GEMM TFLOP/s vs M (% bf16 peak); RMSNorm HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0


# DRAM bytes (read + write) of one gate_up launch at M=8192 from an ncu capture
# of that launch, valid only for the kernel source it was taken on (checked by
# hash at run time).
GATE_UP_TRAFFIC = {"source_sha256_16": "69f9219b446c07e9", "bytes": 887380480 + 386338816}


def gate_up_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_bf16_pair.cu", "bi_ptx.cuh"):
        with open(os.path.join(ROOT, "invariant_deterministic_bi_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return GATE_UP_TRAFFIC["bytes"] if h.hexdigest()[:16] == GATE_UP_TRAFFIC["source_sha256_16"] else None


def step_flops(M: int) -> float:
    return sum(2.0 * M * n * k for n, k in LAYERS.values())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, world, rank, backend):
        self.world, self.rank = world, rank
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bi_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- our arm

def bf16_dev(bits):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def make_step_inputs(M: int, seed: int = 0):
    """Synthetic Qwen3-8B-shaped inputs (bf16, device resident)."""
    import bi_synth as syn
    d = {}
    x, res, w1, _ = syn.rmsnorm_inputs(M, H, seed=seed, outlier_frac=0.0)
    x2, _, w2, _ = syn.rmsnorm_inputs(M, H, seed=seed + 1, outlier_frac=0.0)
    d["x"], d["x2"], d["res"], d["w1"], d["w2"] = map(bf16_dev, (x, x2, res, w1, w2))
    for i, (name, (n, k)) in enumerate(LAYERS.items()):
        d["W_" + name] = bf16_dev(syn.to_bf16_bits(syn.normal_rows(seed + 10 + i, syn.TID_W, n, k, std=0.02)))
    return d


class Step:
    """One pass of the hot path; optional per-GEMM events for the roofline."""

    def __init__(self, bi, inp, M):
        import torch
        self.bi, self.inp, self.M = bi, inp, M
        self.h1 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        self.h2 = torch.empty_like(self.h1)
        self.qkv = torch.empty((M, LAYERS["qkv"][0]), dtype=torch.bfloat16, device="cuda")
        self.gu = torch.empty((M, LAYERS["gate_up"][0]), dtype=torch.bfloat16, device="cuda")
        self.dn = torch.empty((M, LAYERS["down"][0]), dtype=torch.bfloat16, device="cuda")
        self.gemm_events = []

    def __call__(self, events=False):
        import torch
        bi, d = self.bi, self.inp
        ev = (lambda: torch.cuda.Event(enable_timing=True)) if events else None

        def gemm(X, W, Y):
            if events:
                a, b = ev(), ev()
                a.record()
                bi.gemm_bf16(X, W, Y=Y)
                b.record()
                self.gemm_events.append((a, b))
            else:
                bi.gemm_bf16(X, W, Y=Y)

        bi.rmsnorm(d["x"], d["w1"], EPS, residual=d["res"], out=self.h1)
        gemm(self.h1, d["W_qkv"], self.qkv)
        bi.rmsnorm(d["x2"], d["w2"], EPS, residual=d["res"], out=self.h2)
        gemm(self.h2, d["W_gate_up"], self.gu)
        gemm(self.gu[:, :LAYERS["down"][1]], d["W_down"], self.dn)


def time_fn(fn, reps: int, warm: int = 3, graph: bool = True) -> float:
    """Mean device time (ms) of fn() over reps back-to-back calls, CUDA events
    around one replay of a CUDA graph holding the reps calls (so small calls
    are not timed at the host's launch rate). graph=False times eager calls."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if not graph:
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) / reps


def l2_sets(nbytes: float, cap: int = 16) -> int:
    """Input sets to cycle through so that consecutive calls touch more than
    twice the L2 (a call's reads hit L2 only if it ran within the last sets)."""
    import torch
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    return max(1, min(cap, int(2 * l2 // max(1.0, nbytes)) + 1))


def rotate(inputs_list):
    """Cycle through several input sets so consecutive calls miss in L2."""
    state = {"i": 0}

    def nxt():
        v = inputs_list[state["i"] % len(inputs_list)]
        state["i"] += 1
        return v
    return nxt


def gemm_sweep(bi, peaks):
    """TFLOP/s of bi_gemm_bf16 vs M for each layer, against cuBLAS (torch.matmul)."""
    import torch
    import bi_synth as syn
    rows = []
    for name, (n, k) in LAYERS.items():
        W0 = bf16_dev(syn.to_bf16_bits(syn.normal_rows(20, syn.TID_W, n, k, std=0.02)))
        Ws = [W0] + [W0.clone() for _ in range(l2_sets(2.0 * n * k) - 1)]   # weights rotate past L2
        Xmax = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_X, max(M_SWEEP), k)))
        for M in M_SWEEP:
            X = Xmax[:M]
            Y = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
            wsel = rotate(Ws)
            reps = 50 if M <= 513 else 10
            t_bi = time_fn(lambda: bi.gemm_bf16(X, wsel(), Y=Y), reps)
            wsel2 = rotate(Ws)
            t_cb = time_fn(lambda: torch.matmul(X, wsel2().t(), out=Y), reps)
            flops = 2.0 * M * n * k
            tf = flops / (t_bi * 1e-3) / 1e12
            rows.append({"layer": name, "M": M, "N": n, "K": k, "us": round(t_bi * 1e3, 2),
                         "tflops": round(tf, 1), "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 3),
                         "weight_gbs": round(2.0 * n * k / (t_bi * 1e-3) / 1e9, 0),
                         "cublas_us": round(t_cb * 1e3, 2), "cost_vs_cublas": round(t_bi / t_cb, 3)})
        del Ws, Xmax
        torch.cuda.empty_cache()
    # is cuBLAS itself batch-invariant here? (informational)
    n, k = LAYERS["qkv"]
    W = bf16_dev(syn.to_bf16_bits(syn.normal_rows(20, syn.TID_W, n, k, std=0.02)))
    X = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_X, 4096, k)))
    full = torch.matmul(X, W.t())
    one = torch.matmul(X[:1], W.t())
    cublas_inv = bool(torch.equal(full[0], one[0]))
    return rows, cublas_inv


def rmsnorm_sweep(bi, peaks):
    import torch
    import bi_synth as syn
    rows = []
    for with_res in (True, False):
        for M in RMS_SWEEP:
            sets = []
            nsets = l2_sets((8 if with_res else 4) * M * H)
            for j in range(nsets):
                x, res, w, _ = syn.rmsnorm_inputs(M, H, seed=j)
                sets.append((bf16_dev(x), bf16_dev(res) if with_res else None, bf16_dev(w),
                             torch.empty((M, H), dtype=torch.bfloat16, device="cuda")))
            sel = rotate(sets)

            def ours():
                x, r, w, o = sel()
                bi.rmsnorm(x, w, EPS, residual=r, out=o)
            sel2 = rotate(sets)

            def theirs():
                x, r, w, o = sel2()
                if r is not None:
                    r.add_(x)
                    torch.nn.functional.rms_norm(r, (H,), w, EPS)
                else:
                    torch.nn.functional.rms_norm(x, (H,), w, EPS)
            reps = 200 if M <= 128 else 30
            t = time_fn(ours, reps)
            t2 = time_fn(theirs, reps)
            nbytes = (8 if with_res else 4) * M * H + 2 * H
            gbs = nbytes / (t * 1e-3) / 1e9
            rows.append({"M": M, "H": H, "residual": with_res, "us": round(t * 1e3, 2), "gbs": round(gbs, 0),
                         "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3),
                         "frac_hbm_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 3),
                         "torch_us": round(t2 * 1e3, 2), "cost_vs_torch": round(t / t2, 3)})
            del sets
    return rows


RANK_SUM_R = [2, 4, 8]
RANK_SUM_M = [1, 128, 16384]


def rank_sum_sweep(bi, peaks):
    """The tensor-parallel all-reduce + RMSNorm step (bi_rank_sum_rmsnorm) with R
    ranks' partial rows resident on this GPU (as after a gather), residual
    updated in place: HBM bytes = (2R + 6) M H (R parts and the residual read,
    residual and output written)."""
    import torch
    import bi_synth as syn
    rows = []
    for R in RANK_SUM_R:
        for M in RANK_SUM_M:
            nbytes = (2 * R + 6) * M * H
            sets = []
            g = torch.Generator(device="cuda").manual_seed(R * 1000 + M)
            _, _, w, _ = syn.rmsnorm_inputs(1, H, seed=0)
            wd = bf16_dev(w)
            for j in range(l2_sets(nbytes, cap=8)):   # values do not matter for the timing
                parts = [torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16) for _ in range(R)]
                res = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
                sets.append((parts, res, wd, torch.empty((M, H), dtype=torch.bfloat16, device="cuda")))
            sel = rotate(sets)

            def ours():
                parts, res, w, out = sel()
                bi.rank_sum_rmsnorm(parts, w, EPS, residual=res, out=out)
            t = time_fn(ours, 200 if M <= 128 else 30)
            gbs = nbytes / (t * 1e-3) / 1e9
            rows.append({"R": R, "M": M, "H": H, "us": round(t * 1e3, 2), "gbs": round(gbs, 0),
                         "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3)})
            del sets
    return rows


def torch_rmsnorm_row0_equal() -> bool:
    """Informational: is torch.nn.functional.rms_norm batch-invariant here, i.e.
    does row 0 of an M=16384 call equal the same row normalised alone?"""
    import torch
    import bi_synth as syn
    M = max(RMS_SWEEP)
    x, _, w, _ = syn.rmsnorm_inputs(M, H, seed=0)
    xd, wd = bf16_dev(x), bf16_dev(w)
    full = torch.nn.functional.rms_norm(xd, (H,), wd, EPS)
    one = torch.nn.functional.rms_norm(xd[:1].clone(), (H,), wd, EPS)
    torch.cuda.synchronize()
    return bool(torch.equal(full[:1].view(torch.int16), one.view(torch.int16)))


MOE_E, MOE_TOPK = 128, 8
MOE_LAYERS = {"gate_up": (1536, 2048), "down": (2048, 768)}
MOE_T = [1, 64, 512, 8192]


def moe_inputs(layer: str, T: int, seed: int = 0, W=None):
    """Qwen3-30B-A3B-shaped expert inputs: top-8 of 128 experts from seeded
    router logits; rows grouped by expert (device tensors)."""
    import bi_synth as syn
    n, k = MOE_LAYERS[layer]
    tok, exp, off, _ = syn.moe_routing(T, MOE_E, MOE_TOPK, seed=seed)
    if layer == "gate_up":
        X = syn.to_bf16_bits(syn.normal_rows(seed, syn.TID_HIDDEN, T, k))[tok]
    else:
        X = syn.to_bf16_bits(syn.normal_rows(seed, syn.TID_DOWN_IN, T * MOE_TOPK, k))
    if W is None:
        W = bf16_dev(syn.moe_weights(MOE_E, n, k, seed=seed,
                                     tensor_id=syn.TID_W1 if layer == "gate_up" else syn.TID_W2))
    import torch
    return bf16_dev(X), W, torch.from_numpy(off).cuda(), exp


def moe_sweep(bi, peaks):
    """Grouped expert GEMM throughput vs tokens, against torch's grouped GEMM."""
    import torch
    rows = []
    for layer, (n, k) in MOE_LAYERS.items():
        W = None
        for T in MOE_T:
            X, W, off, exp = moe_inputs(layer, T, W=W)
            Y = torch.empty((X.shape[0], n), dtype=torch.bfloat16, device="cuda")
            touched = len(set(exp.tolist()))
            # copies of the expert weights so the touched experts' weights rotate past L2
            Wsets = [W] + [W.clone() for _ in range(l2_sets(2.0 * touched * n * k, cap=6) - 1)]
            wsel = rotate(Wsets)
            t = time_fn(lambda: bi.grouped_gemm_bf16(X, wsel(), off, Y=Y), 20 if T <= 512 else 5)
            flops = 2.0 * X.shape[0] * n * k
            nbytes = 2.0 * (touched * n * k + X.shape[0] * (k + n))
            r = {"layer": layer, "T": T, "rows": int(X.shape[0]), "experts_touched": touched, "us": round(t * 1e3, 2),
                 "tflops": round(flops / (t * 1e-3) / 1e12, 1),
                 "frac_bf16_peak": round(flops / (t * 1e-3) / 1e12 / peaks["bf16_tflops"], 3),
                 "gbs": round(nbytes / (t * 1e-3) / 1e9, 0),
                 "frac_hbm_measured": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
            # non-invariant library reference: one cuBLAS matmul per non-empty expert
            offh = off.cpu().tolist()
            segs = [(e, offh[e], offh[e + 1]) for e in range(MOE_E) if offh[e + 1] > offh[e]]

            wsel2 = rotate(Wsets)

            def per_expert():
                Wc = wsel2()
                for e, a, b in segs:
                    torch.matmul(X[a:b], Wc[e].t(), out=Y[a:b])
            t2 = time_fn(per_expert, 20 if T <= 512 else 5)
            r["cublas_per_expert_us"] = round(t2 * 1e3, 2)
            r["cost_vs_cublas_per_expert"] = round(t / t2, 3)
            r["weight_sets"] = len(Wsets)
            rows.append(r)
            del Wsets
        del W
        torch.cuda.empty_cache()
    return rows


NVFP4_N, NVFP4_K = 14336, 4096
NVFP4_M = [1, 16, 256, 4096]


def torch_nvfp4_mm(A, SA_il, B, SB_il, M, N, K):
    """cuBLASLt NVFP4 GEMM through torch._scaled_mm (not batch-invariant by
    contract); returns a callable, or None when this torch build lacks it."""
    import torch
    try:
        a = A.view(torch.float4_e2m1fn_x2)
        b = B.view(torch.float4_e2m1fn_x2).t()
        rp = lambda r: -(-r // 128) * 128
        cp = -(-(K // 16) // 4) * 4
        sa = SA_il.view(torch.float8_e4m3fn)[: rp(M) * cp].view(rp(M), cp)
        sb = SB_il.view(torch.float8_e4m3fn)[: rp(N) * cp].view(rp(N), cp)
        fn = lambda: torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
    except Exception:
        return None
    try:
        fn()
    except RuntimeError:     # argument rejected on the host: not available here
        return None
    torch.cuda.synchronize()  # a device error here is not swallowed
    return fn


def nvfp4_sweep(bi, peaks):
    """bi_gemm_nvfp4 vs M at K=4096, N=14336, against cuBLASLt NVFP4 via torch."""
    import torch
    import bi_synth as syn
    d = syn.nvfp4_inputs(max(NVFP4_M), NVFP4_N, NVFP4_K, seed=0)
    Bd, SBd = torch.from_numpy(d["B"]).cuda(), torch.from_numpy(d["SB_il"]).cuda()
    bsets = [(Bd, SBd)] + [(Bd.clone(), SBd.clone())
                           for _ in range(l2_sets(Bd.numel() + SBd.numel()) - 1)]   # weights rotate past L2
    rows, fp4_peak, peak_note = [], None, "unmeasured"
    # dense fp4 peak on this GPU: cuBLASLt NVFP4 at 8192^3, if torch exposes it
    use_lt = os.environ.get("BI_BENCH_CUBLASLT_FP4", "1") == "1"
    if use_lt:
        g = torch.Generator(device="cuda").manual_seed(0)
        big = torch.randint(0, 256, (8192, 4096), dtype=torch.uint8, device="cuda", generator=g)
        sc = torch.full((8192 * 512,), 0x38, dtype=torch.uint8, device="cuda")
        f = torch_nvfp4_mm(big, sc, big, sc, 8192, 8192, 8192)
        if f is not None:
            t = time_fn(f, 20)
            fp4_peak = 2.0 * 8192 ** 3 / (t * 1e-3) / 1e12
            peak_note = "measured: cuBLASLt NVFP4 8192^3 via torch._scaled_mm (burst)"
        del big, sc
    if fp4_peak is None:
        fp4_peak = peaks["bf16_tflops"] * 6.0
        peak_note = "measured bf16 peak x 6 (nominal fp4/bf16 dense ratio 13.5/2.25)"
    for M in NVFP4_M:
        A = torch.from_numpy(d["A"][:M].copy()).cuda()
        SA = torch.from_numpy(syn.swizzle_block_scales(d["SA"][:M])).cuda()
        Y = torch.empty((M, NVFP4_N), dtype=torch.bfloat16, device="cuda")
        bsel = rotate(bsets)
        t = time_fn(lambda: bi.gemm_nvfp4(A, SA, *bsel(), float(d["alpha"]), Y=Y), 50 if M <= 256 else 10)
        flops = 2.0 * M * NVFP4_N * NVFP4_K
        nbytes = (M + NVFP4_N) * NVFP4_K * (0.5 + 1 / 16) + 2 * M * NVFP4_N
        r = {"M": M, "N": NVFP4_N, "K": NVFP4_K, "us": round(t * 1e3, 2),
             "tflops": round(flops / (t * 1e-3) / 1e12, 1),
             "frac_fp4_peak": round(flops / (t * 1e-3) / 1e12 / fp4_peak, 3),
             "gbs": round(nbytes / (t * 1e-3) / 1e9, 0),
             "frac_hbm_measured": round(nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
        f = torch_nvfp4_mm(A, SA, Bd, SBd, M, NVFP4_N, NVFP4_K) if use_lt \
            else None
        if f is not None:
            t2 = time_fn(f, 50 if M <= 256 else 10)
            r["cublaslt_us"] = round(t2 * 1e3, 2)
            r["cost_vs_cublaslt"] = round(t / t2, 3)
            ours = Y.float()
            theirs = f().float() * float(d["alpha"])
            r["max_rel_diff_vs_cublaslt"] = float(((ours - theirs).abs() / (theirs.abs() + 1)).max())
        rows.append(r)
    # is cuBLASLt's NVFP4 GEMM itself batch-invariant here? (informational)
    lt_inv = None
    if use_lt:
        Mx = max(NVFP4_M)
        A = torch.from_numpy(d["A"][:Mx].copy()).cuda()
        SA = torch.from_numpy(syn.swizzle_block_scales(d["SA"][:Mx])).cuda()
        A1 = torch.from_numpy(d["A"][:1].copy()).cuda()
        SA1 = torch.from_numpy(syn.swizzle_block_scales(d["SA"][:1])).cuda()
        f_full = torch_nvfp4_mm(A, SA, Bd, SBd, Mx, NVFP4_N, NVFP4_K)
        f_one = torch_nvfp4_mm(A1, SA1, Bd, SBd, 1, NVFP4_N, NVFP4_K)
        if f_full is not None and f_one is not None:
            lt_inv = bool(torch.equal(f_full()[0], f_one()[0]))
    return {"fp4_peak_tflops": round(fp4_peak, 1), "fp4_peak_source": peak_note, "rows": rows,
            "cublaslt_row0_equal_M1_vs_M4096": lt_inv}


QUANT_M = [1, 16, 256, 4096, 16384]


def quant_sweep(bi, peaks):
    """bi_quantize_nvfp4 at K=4096: HBM GB/s (reads 2 B, writes 0.5 + 1/16 B per element)."""
    import torch
    import bi_synth as syn
    K = NVFP4_K
    rows = []
    for M in QUANT_M:
        nsets = l2_sets(M * K * (2 + 0.5 + 1 / 16))
        sets = []
        for j in range(nsets):
            X = bf16_dev(syn.to_bf16_bits(syn.normal_rows(j, syn.TID_FP4_A, M, K)))
            Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
            S = torch.zeros(-(-M // 128) * 128 * (K // 16), dtype=torch.uint8, device="cuda")
            sets.append((X, Q, S))
        sel = rotate(sets)

        def call():
            X, Q, S = sel()
            bi.quantize_nvfp4(X, 1.0, Q=Q, Q_sf=S)
        t = time_fn(call, 200 if M <= 256 else 30)
        nbytes = M * K * (2 + 0.5 + 1 / 16)
        gbs = nbytes / (t * 1e-3) / 1e9
        rows.append({"M": M, "K": K, "us": round(t * 1e3, 2), "gbs": round(gbs, 0),
                     "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3)})
        del sets
    return rows


MOE_LAYER_T = [1, 64, 512, 8192]


def moe_layer_sweep(bi, peaks):
    """The whole batch-invariant MoE layer (Qwen3-30B-A3B shapes): router top-8
    softmax, alignment, gather, grouped gate_up, SiLU-mul, grouped down,
    rank-order combine. Per-stage device time (CUDA-graph replays), and the
    layer with gate_up and SiLU-mul fused (checked bit-equal to the pair)."""
    import torch
    import bi_synth as syn
    n1, k1 = MOE_LAYERS["gate_up"]
    n2, k2 = MOE_LAYERS["down"]
    W1 = bf16_dev(syn.moe_weights(MOE_E, n1, k1, seed=0, tensor_id=syn.TID_W1))
    W2 = bf16_dev(syn.moe_weights(MOE_E, n2, k2, seed=0, tensor_id=syn.TID_W2))
    out = []
    for T in MOE_LAYER_T:
        hidden = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_HIDDEN, T, k1)))
        logits = torch.from_numpy(syn.normal_rows(0, syn.TID_LOGITS, T, MOE_E)).cuda()
        ids, w = bi.moe_topk_softmax(logits, MOE_TOPK)
        off, rt, pos = bi.moe_align(ids, MOE_E)
        X = bi.moe_gather(hidden, rt)
        gu = bi.grouped_gemm_bf16(X, W1, off)
        act = bi.silu_mul(gu)
        y = bi.grouped_gemm_bf16(act, W2, off)
        o = bi.moe_combine(y, pos, w)
        act_f = bi.grouped_gemm_silu_bf16(X, W1, off)
        if not torch.equal(act_f.view(torch.int16), act.view(torch.int16)):
            raise RuntimeError(f"fused gate_up + SiLU-mul differs from the unfused pair at T={T}")
        # the experts' weights come from HBM, as in a model whose layers each
        # have their own: at small T the touched experts would fit in L2, so
        # the weights rotate over copies
        touched = int((off[1:] - off[:-1] > 0).sum().item())
        nsets = l2_sets(2.0 * touched * (n1 * k1 + n2 * k2), cap=6)
        W1s = [W1] + [W1.clone() for _ in range(nsets - 1)]
        W2s = [W2] + [W2.clone() for _ in range(nsets - 1)]
        w1a, w1b, w2a = rotate(W1s), rotate(W1s), rotate(W2s)
        reps = 50 if T <= 512 else 10
        stages = {
            "topk_softmax": lambda: bi.moe_topk_softmax(logits, MOE_TOPK),
            "align": lambda: bi.moe_align(ids, MOE_E),
            "gather": lambda: bi.moe_gather(hidden, rt, out=X),
            "grouped_gate_up": lambda: bi.grouped_gemm_bf16(X, w1a(), off, Y=gu),
            "silu_mul": lambda: bi.silu_mul(gu, out=act),
            "grouped_down": lambda: bi.grouped_gemm_bf16(act, w2a(), off, Y=y),
            "combine": lambda: bi.moe_combine(y, pos, w, out=o),
        }
        times = {name: round(time_fn(fn, reps) * 1e3, 2) for name, fn in stages.items()}
        fused_us = round(time_fn(lambda: bi.grouped_gemm_silu_bf16(X, w1b(), off, act=act_f), reps) * 1e3, 2)
        total_us = sum(times.values())
        total_fused = total_us - times["grouped_gate_up"] - times["silu_mul"] + fused_us
        flops = 2.0 * T * MOE_TOPK * (n1 * k1 + n2 * k2)
        out.append({"T": T, "us_by_stage": times, "us_total": round(total_us, 2),
                    "gemm_share": round((times["grouped_gate_up"] + times["grouped_down"]) / total_us, 3),
                    "tflops_layer": round(flops / (total_us * 1e-6) / 1e12, 1),
                    "fused_gate_up_silu_us": fused_us, "us_total_fused": round(total_fused, 2),
                    "tflops_layer_fused": round(flops / (total_fused * 1e-6) / 1e12, 1),
                    "weight_sets": nsets})
        del hidden, logits, ids, w, off, rt, pos, X, gu, act, act_f, y, o, W1s, W2s
    del W1, W2
    torch.cuda.empty_cache()
    return out


ATTN_B = [1, 8, 64]
ATTN_L = 4096
ATTN_HEADS = (32, 8, 128, 16)     # Qwen3-8B: query heads, KV heads, head_dim; KV block size


def attention_sweep(bi, peaks):
    """Decode attention, Qwen3-8B heads (32 q, 8 kv, dim 128), paged KV (block 16),
    every sequence 4096 tokens: KV GB/s against HBM (KV bytes dominate)."""
    import torch
    Hq, Hkv, D, bs = ATTN_HEADS
    rows = []
    g = torch.Generator(device="cuda").manual_seed(0)
    for B in ATTN_B:
        nb = ATTN_L // bs
        blocks = B * nb
        K = torch.randn((blocks, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        V = torch.randn((blocks, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        table = torch.randperm(blocks, device="cuda", generator=g).to(torch.int32).view(B, nb)
        lens = torch.full((B,), ATTN_L, dtype=torch.int32, device="cuda")
        Q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        ws = torch.empty(bi.attention_decode_workspace_size(B, Hq, ATTN_L), dtype=torch.uint8, device="cuda")
        O = torch.empty_like(Q)
        kvsets = [(K, V)] + [(K.clone(), V.clone()) for _ in range(l2_sets(2.0 * K.numel() * 2) - 1)]
        kvsel = rotate(kvsets)             # the KV cache rotates past L2

        def call():
            Kc, Vc = kvsel()
            bi.attention_decode(Q, Kc, Vc, table, lens, ATTN_L, D ** -0.5, workspace=ws, O=O)
        t = time_fn(call, 50 if B <= 8 else 10)
        kv_bytes = 2.0 * B * ATTN_L * Hkv * D * 2
        gbs = kv_bytes / (t * 1e-3) / 1e9
        rows.append({"B": B, "L": ATTN_L, "us": round(t * 1e3, 2), "kv_gbs": round(gbs, 0),
                     "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3)})
        del K, V, kvsets, table, lens, Q, ws, O
    torch.cuda.empty_cache()
    return rows


EXT_CASES = [(1, 4096, 4096), (8, 512, 512), (4, 1024, 4096)]   # (sequences, new tokens each, cached length each)


def extend_flops(q, L):
    """Causal attention FLOPs of q new tokens ending a length-L cache, per query head:
    token at position p costs 2*2*D*(p+1) (q.k and p.v)."""
    D = ATTN_HEADS[2]
    first = L - q
    return 4.0 * D * (q * (first + 1) + q * (q - 1) / 2.0)


def extend_sweep(bi, peaks):
    """Extend (prefill) attention, Qwen3-8B heads, paged KV (block 16): TFLOP/s
    of the causal attention, against torch's scaled_dot_product_attention on
    the same data laid out contiguously (not paged, not batch-invariant;
    informational)."""
    import torch
    Hq, Hkv, D, bs = ATTN_HEADS
    rows = []
    g = torch.Generator(device="cuda").manual_seed(0)
    for B, q, L in EXT_CASES:
        nb = L // bs
        K = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        V = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        table = torch.randperm(B * nb, device="cuda", generator=g).to(torch.int32).view(B, nb)
        lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
        cu = torch.arange(0, (B + 1) * q, q, dtype=torch.int32, device="cuda")
        Q = torch.randn((B * q, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        O = torch.empty_like(Q)
        t = time_fn(lambda: bi.attention_extend(Q, cu, K, V, table, lens, L, q, D ** -0.5, O=O), 10)
        flops = B * Hq * extend_flops(q, L)
        row = {"B": B, "new_tokens": q, "cached": L, "us": round(t * 1e3, 2), "tflops": round(flops / (t * 1e-3) / 1e12, 1)}
        try:     # the same attention by torch on contiguous K/V (causal with an offset: an explicit mask)
            kc = K[table.view(-1).long()].view(B, L, Hkv, D).permute(0, 2, 1, 3).contiguous()
            vc = V[table.view(-1).long()].view(B, L, Hkv, D).permute(0, 2, 1, 3).contiguous()
            qc = Q.view(B, q, Hq, D).permute(0, 2, 1, 3).contiguous()
            sdpa = torch.nn.functional.scaled_dot_product_attention
            if q == L:    # plain causal: torch may use its flash kernel
                mask = None
                t2 = time_fn(lambda: sdpa(qc, kc, vc, is_causal=True, scale=D ** -0.5, enable_gqa=True), 10)
            else:         # causal with an offset needs an explicit mask
                pos = torch.arange(L - q, L, device="cuda")[:, None]
                mask = torch.arange(L, device="cuda")[None, :] <= pos
                t2 = time_fn(lambda: sdpa(qc, kc, vc, attn_mask=mask, scale=D ** -0.5, enable_gqa=True), 10)
            row["torch_sdpa_us"] = round(t2 * 1e3, 2)
            row["torch_sdpa_form"] = "is_causal" if mask is None else "explicit mask"
            row["cost_vs_torch_sdpa"] = round(t / t2, 3)
            del kc, vc, qc, mask
        except (RuntimeError, TypeError) as exc:      # no GQA support in this torch: leave it out
            if "CUDA" in str(exc) and "error" in str(exc).lower():
                raise
            row["torch_sdpa_us"] = None
        rows.append(row)
        del K, V, table, lens, cu, Q, O
    torch.cuda.empty_cache()
    return rows


_STEP_WEIGHTS = {}


def step_weights():
    """The step's three weight matrices as bf16 bits (seeded; generated once)."""
    import bi_synth as syn
    if not _STEP_WEIGHTS:
        for i, (name, (n, k)) in enumerate(LAYERS.items()):
            _STEP_WEIGHTS[name] = syn.to_bf16_bits(syn.normal_rows(10 + i, syn.TID_W, n, k, std=0.02))
    return _STEP_WEIGHTS


def cpu_baseline(rows: int):
    """The fp64 oracle on a bounded sample of the step: `rows` rows of every
    GEMM of the step and of both RMSNorms, on the host's cores."""
    import numpy as np
    import bi_synth as syn
    import oracle
    x, res, w, _ = syn.rmsnorm_inputs(rows, H, seed=0, outlier_frac=0.0)
    Ws = step_weights()
    Xd = syn.to_bf16_bits(syn.normal_rows(0, syn.TID_X, rows, LAYERS["down"][1]))
    t0 = time.perf_counter()
    y1, h = oracle.rmsnorm(x, w, EPS, residual=res)
    oracle.gemm_bf16(oracle.bf16_round_array(y1), Ws["qkv"])
    y2, _ = oracle.rmsnorm(x, w, EPS, residual=h)
    oracle.gemm_bf16(oracle.bf16_round_array(y2), Ws["gate_up"])
    oracle.gemm_bf16(Xd, Ws["down"])
    dt = time.perf_counter() - t0
    return step_flops(rows) / dt / 1e12, dt, oracle.threads()


def e2e_pipelined(bi, inp, M: int, k: int, dist, nslots: int = 3):
    """The step end to end from pinned host memory: every step copies its three
    activation inputs (x, x2, residual) host -> device and its two results
    (qkv and down outputs) device -> host. `nslots` device buffer sets let
    later steps' inputs and earlier steps' results move on their own streams
    while a step computes; with three, a step's compute never waits for the
    results of the step before last to leave its buffers. Returns (ms per step
    over k steps, H2D bytes, D2H bytes per step)."""
    import torch
    names = ("x", "x2", "res")
    host_in = {n: torch.empty_like(inp[n], device="cpu").pin_memory() for n in names}
    for n in names:
        host_in[n].copy_(inp[n].cpu())
    slots = []
    for _ in range(nslots):
        d = dict(inp)
        for n in names:
            d[n] = torch.empty_like(inp[n])
        st = Step(bi, d, M)
        hq = torch.empty_like(st.qkv, device="cpu").pin_memory()
        hd = torch.empty_like(st.dn, device="cpu").pin_memory()
        ev = {e: torch.cuda.Event() for e in ("in_done", "comp_done", "out_done")}
        slots.append((d, st, hq, hd, ev))
    s_c = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def one(i):
        d, st, hq, hd, ev = slots[i % nslots]
        with torch.cuda.stream(s_in):
            if i >= nslots:
                s_in.wait_event(ev["comp_done"])      # slot's inputs no longer read
            for n in names:
                d[n].copy_(host_in[n], non_blocking=True)
            ev["in_done"].record(s_in)
        s_c.wait_event(ev["in_done"])
        if i >= nslots:
            s_c.wait_event(ev["out_done"])            # slot's results already copied out
        st()
        ev["comp_done"].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp_done"])
            hq.copy_(st.qkv, non_blocking=True)
            hd.copy_(st.dn, non_blocking=True)
            ev["out_done"].record(s_out)

    for i in range(nslots):                            # warm-up
        one(i)
    torch.cuda.synchronize()
    dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_c)
    s_in.wait_stream(s_c)                              # first copy starts after the start mark
    for i in range(k):
        one(i)
    s_c.wait_stream(s_out)                             # last results are on the host
    b.record(s_c)
    torch.cuda.synchronize()
    ms = dist.max(a.elapsed_time(b)) / k
    h2d = sum(inp[n].numel() for n in names) * 2
    d2h = (slots[0][1].qkv.numel() + slots[0][1].dn.numel()) * 2
    return ms, h2d, d2h


def step_config(world: int) -> dict:
    """The workload both arms report (the reference arm times a row sample of it)."""
    return {"workload": "Qwen3-8B-shaped decoder-layer linears at M=8192: RMSNorm+residual -> qkv "
                        "(4096->6144) -> RMSNorm+residual -> gate_up (4096->24576) -> down (12288->4096)",
            "M": M_STEP, "hidden": H, "parallelism": f"replicas x{world}",
            "l2": "no flush: each step streams > 1 GB (weights 352 MB + activations), L2 is 129 MB"}


def run_ours(args, dist):
    import torch
    import invariant_deterministic_bi_gb300 as bi
    bi.load()
    peaks, peak_src = load_peaks()
    M = M_STEP
    inp = make_step_inputs(M, seed=dist.rank)
    step = Step(bi, inp, M)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = bi.device_status()
    if st != bi.BI_OK:
        raise RuntimeError(f"device status after warm-up: {bi.status_string(st)}")

    # ---- timed region: K steps back to back, events around each GEMM launch
    dist.barrier()
    torch.cuda.synchronize()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0e.record()
        for _ in range(args.steps):
            step(events=True)
        t1e.record()
        torch.cuda.synchronize()
    dist.barrier()
    ms_total = dist.max(t0e.elapsed_time(t1e))
    clocks = clk.summary()
    gemm_ms = [a.elapsed_time(b) for a, b in step.gemm_events]
    st = bi.device_status()
    if st != bi.BI_OK:
        raise RuntimeError(f"device status after timed steps: {bi.status_string(st)}")

    ms_per_step = ms_total / args.steps
    flops = step_flops(M)
    value = flops * dist.world / (ms_per_step * 1e-3) / 1e12
    launches_per_step = 5
    # dominant kernel: the gate_up launch of bi_gemm_bf16 (the largest of the step)
    per = {}
    for i, name in enumerate(LAYERS):
        ms_i = gemm_ms[i::3]
        n, k = LAYERS[name]
        per[name] = round(2.0 * M * n * k / (sum(ms_i) / len(ms_i) * 1e-3) / 1e12, 1)
    achieved = per["gate_up"]
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    capped = "sw_power_cap" in clocks.get("reasons", [])
    peak = sustained if capped else burst
    roofline = {"kernel": "bi_gemm_bf16 gate_up launch (M=8192, N=24576, K=4096)", "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 3),
                "peak_source": (f"{peak_src} bf16 sustained (cuBLAS 8192^3 back to back under the power cap): "
                                "sw_power_cap was active during the timed steps") if capped else
                               (f"{peak_src} bf16 burst (cuBLAS 8192^3, best of 10): no power cap was "
                                "active during the timed steps"),
                "frac_of_burst_peak": round(achieved / burst, 3),
                "frac_of_sustained_peak": round(achieved / sustained, 3),
                "step_frac_of_burst_peak": round(flops / (ms_per_step * 1e-3) / 1e12 / burst, 3),
                "achieved_per_layer": per,
                "algorithmic_bytes": int(2 * (M * 4096 + 24576 * 4096 + M * 24576)),
                "traffic": gate_up_traffic()}
    for name, v in per.items():
        roofline[f"step_{name}_tflops"] = v

    # ---- end to end: host buffers in, results out, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        ms, h2d, d2h = e2e_pipelined(bi, inp, M, max(10, args.steps), dist)
        e2e = {"value": round(flops * dist.world / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
               "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelining": "3 buffer sets; later steps' host-to-device copies and earlier steps' "
                             "device-to-host copies run on their own streams while a step computes; the "
                             "host link moves ~200 GB/s each way, ~320 GB/s with both directions at once"}

    breakdown = {}
    if not args.no_breakdown and dist.rank == 0:
        rows, cublas_inv = gemm_sweep(bi, peaks)
        breakdown["gemm_bf16_vs_M"] = rows
        breakdown["cublas_row0_equal_M1_vs_M4096"] = cublas_inv
        breakdown["rmsnorm"] = rmsnorm_sweep(bi, peaks)
        breakdown["torch_rms_norm_row0_equal_M1_vs_M16384"] = torch_rmsnorm_row0_equal()
        breakdown["rank_sum_rmsnorm"] = rank_sum_sweep(bi, peaks)
        breakdown["grouped_gemm_bf16_moe"] = moe_sweep(bi, peaks)
        breakdown["gemm_nvfp4"] = nvfp4_sweep(bi, peaks)
        breakdown["quantize_nvfp4"] = quant_sweep(bi, peaks)
        breakdown["moe_layer"] = moe_layer_sweep(bi, peaks)
        breakdown["attention_decode"] = attention_sweep(bi, peaks)
        breakdown["attention_extend"] = extend_sweep(bi, peaks)
        if bi.device_status() != bi.BI_OK:
            raise RuntimeError("device status after breakdown")
        # the metric's per-M GEMM fractions and its RMSNorm half as flat numbers
        for r in breakdown["gemm_bf16_vs_M"]:
            if r["M"] in (1, 7, 64, 4096, 8192):
                key = f"gemm_{r['layer']}_M{r['M']}"
                roofline[key + "_tflops"] = r["tflops"]
                roofline[key + "_frac_bf16_peak"] = r["frac_bf16_peak"]
                roofline[key + "_cost_vs_cublas"] = r["cost_vs_cublas"]
                if r["M"] <= 64:
                    roofline[key + "_weight_frac_hbm"] = round(r["weight_gbs"] / peaks["hbm_gbs"], 3)
        for r in breakdown["rmsnorm"]:
            if r["M"] == max(RMS_SWEEP):
                key = "rmsnorm_M%d_H%d_%s" % (r["M"], r["H"], "res" if r["residual"] else "nores")
                roofline[key + "_gbs"] = r["gbs"]
                roofline[key + "_frac_hbm_measured"] = r["frac_hbm_measured"]
                roofline[key + "_frac_hbm_nominal_8tbs"] = r["frac_hbm_nominal_8tbs"]
                roofline[key + "_us"] = r["us"]
            elif r["M"] == 1:                       # one decode token: latency
                roofline["rmsnorm_M1_H%d_%s_us" % (r["H"], "res" if r["residual"] else "nores")] = r["us"]
        # the other hot-path rows' headline figures, also as flat numbers
        for r in breakdown["gemm_nvfp4"]["rows"]:
            if r["M"] in (1, 4096):
                roofline[f"nvfp4_M{r['M']}_us"] = r["us"]
                roofline[f"nvfp4_M{r['M']}_tflops"] = r["tflops"]
                if "cost_vs_cublaslt" in r:
                    roofline[f"nvfp4_M{r['M']}_cost_vs_cublaslt"] = r["cost_vs_cublaslt"]
        qmax = max(x["M"] for x in breakdown["quantize_nvfp4"])
        for r in breakdown["quantize_nvfp4"]:
            if r["M"] == qmax:
                roofline[f"quantize_nvfp4_M{r['M']}_us"] = r["us"]
                roofline[f"quantize_nvfp4_M{r['M']}_frac_hbm_measured"] = r["frac_hbm_measured"]
        for r in breakdown["rank_sum_rmsnorm"]:
            if r["M"] == max(RANK_SUM_M) and r["R"] == 4:
                roofline["rank_sum_rmsnorm_R4_M%d_us" % r["M"]] = r["us"]
                roofline["rank_sum_rmsnorm_R4_M%d_frac_hbm_measured" % r["M"]] = r["frac_hbm_measured"]
            elif r["M"] == 1 and r["R"] == 4:
                roofline["rank_sum_rmsnorm_R4_M1_us"] = r["us"]
        for r in breakdown["moe_layer"]:
            roofline[f"moe_layer_T{r['T']}_us_fused"] = r["us_total_fused"]
            roofline[f"moe_layer_T{r['T']}_us_unfused"] = r["us_total"]
        for r in breakdown["attention_decode"]:
            roofline[f"attention_decode_B{r['B']}_L{r['L']}_us"] = r["us"]
            roofline[f"attention_decode_B{r['B']}_L{r['L']}_frac_hbm_measured"] = r["frac_hbm_measured"]
        for r in breakdown["attention_extend"]:
            key = f"attention_extend_{r['B']}x{r['new_tokens']}_cached{r['cached']}"
            roofline[key + "_us"] = r["us"]
            roofline[key + "_tflops"] = r["tflops"]

    cpu = None
    if dist.rank == 0 and not args.no_cpu:
        v, dt, cores = cpu_baseline(args.cpu_rows)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{args.cpu_rows} rows of the step (2 RMSNorm rows + qkv/gate_up/down GEMM rows), "
                         f"fp64, {dt:.1f} s"}
        # the same oracle on one core, on a 16-row slice of the step
        import oracle
        oracle.set_threads(1)
        try:
            v1, dt1, _ = cpu_baseline(16)
        finally:
            oracle.set_threads(cores)
        cpu["one_core"] = {"value": round(v1, 6), "unit": "TFLOP/s", "cores": 1,
                           "sample": f"16 rows of the step, fp64, {dt1:.1f} s"}

    # breakdown first, the headline objects last (a truncated tail of the line keeps them)
    line = {"breakdown": breakdown, "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights; no model weights)",
            "config": step_config(dist.world),
            "gpu_launches": launches_per_step * args.steps, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "roofline": roofline}
    return line


# ------------------------------------------------------------ reference arm

def run_reference(args, dist):
    """The fp64 CPU oracle timed as the reference arm, on a bounded sample per step."""
    if dist.rank != 0:
        return None
    rows = args.ref_rows
    for _ in range(args.warmup):
        cpu_baseline(rows)
    t = 0.0
    for _ in range(args.steps):
        _, dt, cores = cpu_baseline(rows)
        t += dt
    ms = t / args.steps * 1e3
    v = step_flops(rows) / (ms * 1e-3) / 1e12
    sample = (f"{rows} of the step's {M_STEP} rows per step (both RMSNorms and the qkv, gate_up and down GEMM rows), "
              f"fp64, OpenMP over rows on {cores} host threads; value = the step's GEMM FLOPs for those rows / time")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(dist.world),
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(spec: str, reps: int):
    """Run one kernel configuration `reps` times (for ncu captures); no output line.
    spec: gemm:<qkv|gate_up|down>:<M> | rmsnorm:<M>:<0|1 residual> | grouped:<gate_up|down>:<T> |
          nvfp4:<M> | quant:<M> | attention:<B> (decode, 4096 cached tokens per sequence) |
          rank_sum:<R>:<M> (all-reduce + RMSNorm over R resident parts) |
          moe_layer:<T> (the whole MoE layer, gate_up with SiLU-mul fused) |
          extend:<B>:<new tokens>:<cached> (prefill attention)"""
    import torch
    import bi_synth as syn
    import invariant_deterministic_bi_gb300 as bi
    bi.load()
    kind, *rest = spec.split(":")
    if kind == "gemm":
        n, k = LAYERS[rest[0]]
        M = int(rest[1])
        X = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_X, M, k)))
        W = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_W, n, k, std=0.02)))
        Y = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
        fn = lambda: bi.gemm_bf16(X, W, Y=Y)
    elif kind == "rmsnorm":
        M, res = int(rest[0]), rest[1] == "1"
        x, r, w, _ = syn.rmsnorm_inputs(M, H, seed=0)
        xd, rd, wd = bf16_dev(x), (bf16_dev(r) if res else None), bf16_dev(w)
        out = torch.empty_like(xd)
        fn = lambda: bi.rmsnorm(xd, wd, EPS, residual=rd, out=out)
    elif kind == "rank_sum":
        R, M = int(rest[0]), int(rest[1])
        g = torch.Generator(device="cuda").manual_seed(0)
        parts = [torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16) for _ in range(R)]
        rd = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
        wd = bf16_dev(syn.rmsnorm_inputs(1, H, seed=0)[2])
        out = torch.empty_like(rd)
        fn = lambda: bi.rank_sum_rmsnorm(parts, wd, EPS, residual=rd, out=out)
    elif kind == "nvfp4":
        M = int(rest[0])
        d = syn.nvfp4_inputs(M, NVFP4_N, NVFP4_K, seed=0)
        A, SA = torch.from_numpy(d["A"]).cuda(), torch.from_numpy(d["SA_il"]).cuda()
        B, SB = torch.from_numpy(d["B"]).cuda(), torch.from_numpy(d["SB_il"]).cuda()
        Y = torch.empty((M, NVFP4_N), dtype=torch.bfloat16, device="cuda")
        fn = lambda: bi.gemm_nvfp4(A, SA, B, SB, float(d["alpha"]), Y=Y)
    elif kind == "quant":
        M = int(rest[0])
        X = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_FP4_A, M, NVFP4_K)))
        Q = torch.empty((M, NVFP4_K // 2), dtype=torch.uint8, device="cuda")
        S = torch.zeros(-(-M // 128) * 128 * (NVFP4_K // 16), dtype=torch.uint8, device="cuda")
        fn = lambda: bi.quantize_nvfp4(X, 1.0, Q=Q, Q_sf=S)
    elif kind == "grouped":
        X, W, off, _ = moe_inputs(rest[0], int(rest[1]))
        Y = torch.empty((X.shape[0], W.shape[1]), dtype=torch.bfloat16, device="cuda")
        fn = lambda: bi.grouped_gemm_bf16(X, W, off, Y=Y)
    elif kind == "moe_layer":
        T = int(rest[0])
        n1, k1 = MOE_LAYERS["gate_up"]
        n2, k2 = MOE_LAYERS["down"]
        W1 = bf16_dev(syn.moe_weights(MOE_E, n1, k1, seed=0, tensor_id=syn.TID_W1))
        W2 = bf16_dev(syn.moe_weights(MOE_E, n2, k2, seed=0, tensor_id=syn.TID_W2))
        hidden = bf16_dev(syn.to_bf16_bits(syn.normal_rows(0, syn.TID_HIDDEN, T, k1)))
        logits = torch.from_numpy(syn.normal_rows(0, syn.TID_LOGITS, T, MOE_E)).cuda()

        def fn():
            ids, w = bi.moe_topk_softmax(logits, MOE_TOPK)
            off, rt, pos = bi.moe_align(ids, MOE_E)
            X = bi.moe_gather(hidden, rt)
            act = bi.grouped_gemm_silu_bf16(X, W1, off)
            y = bi.grouped_gemm_bf16(act, W2, off)
            return bi.moe_combine(y, pos, w)
    elif kind == "attention":
        B, (Hq, Hkv, D, bs) = int(rest[0]), ATTN_HEADS
        nb = ATTN_L // bs
        g = torch.Generator(device="cuda").manual_seed(0)
        K = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        V = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        table = torch.randperm(B * nb, device="cuda", generator=g).to(torch.int32).view(B, nb)
        lens = torch.full((B,), ATTN_L, dtype=torch.int32, device="cuda")
        Q = torch.randn((B, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        ws = torch.empty(bi.attention_decode_workspace_size(B, Hq, ATTN_L), dtype=torch.uint8, device="cuda")
        O = torch.empty_like(Q)
        fn = lambda: bi.attention_decode(Q, K, V, table, lens, ATTN_L, D ** -0.5, workspace=ws, O=O)
    elif kind == "extend":
        B, q, L = (int(v) for v in rest)
        Hq, Hkv, D, bs = ATTN_HEADS
        nb = -(-L // bs)
        g = torch.Generator(device="cuda").manual_seed(0)
        K = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        V = torch.randn((B * nb, bs, Hkv, D), device="cuda", generator=g).to(torch.bfloat16)
        table = torch.randperm(B * nb, device="cuda", generator=g).to(torch.int32).view(B, nb)
        lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
        cu = torch.arange(0, (B + 1) * q, q, dtype=torch.int32, device="cuda")
        Q = torch.randn((B * q, Hq, D), device="cuda", generator=g).to(torch.bfloat16)
        O = torch.empty_like(Q)
        fn = lambda: bi.attention_extend(Q, cu, K, V, table, lens, L, q, D ** -0.5, O=O)
    else:
        raise SystemExit(f"unknown profile case {spec}")
    ms = time_fn(fn, reps, warm=1)
    print(json.dumps({"profile": spec, "reps": reps, "us_per_call": round(ms * 1e3, 2)}), flush=True)
    st = bi.device_status()
    if st != bi.BI_OK:
        raise SystemExit(f"device status {bi.status_string(st)}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=192)
    ap.add_argument("--ref-rows", type=int, default=32)
    ap.add_argument("--profile", default=None, help="run one kernel case only (see profile_case)")
    ap.add_argument("--reps", type=int, default=4)
    args = ap.parse_args()
    if args.profile:
        profile_case(args.profile, args.reps)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank != 0:          # the CPU oracle runs once, on rank 0
            return
        line = run_reference(args, Dist(1, 0, None))
        line["n_gpus"] = world
        print(json.dumps(line), flush=True)
        return
    import torch
    torch.cuda.set_device(local)
    dist = Dist(world, rank, "nccl")
    line = run_ours(args, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
