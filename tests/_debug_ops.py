"""Runs one seeded call of every kernel family on the GPU and prints a digest
of each output and the final device status, one JSON line. The debug-build
test runs it twice, with the release library and with the bounds-checked
debug library (BI_LIBRARY=debug), and compares the digests: the checks may
not change any bit. Not collected by pytest (helper script)."""
import hashlib
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import bi_synth as syn  # noqa: E402
import invariant_deterministic_bi_gb300 as bi  # noqa: E402


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def digest(t):
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()[:16]


def main():
    bi.load()
    out = {"debug_build": bi.debug_build()}
    # dense bf16: one segment, the cluster schedule (M <= 256), one pair per tile with segments
    for name, (M, N, K) in {"gemm_small": (70, 512, 256), "gemm_qkv_m7": (7, 6144, 4096),
                            "gemm_qkv_m300": (300, 6144, 4096), "gemm_down_m5": (5, 4096, 12288)}.items():
        X, W = syn.gemm_inputs(M, N, K, seed=1)
        out[name] = digest(bi.gemm_bf16(dev(X), dev(W)))
    # grouped, with SiLU-mul fused
    off = syn.offsets_from_counts([3, 0, 300, 5])
    Xg = syn.to_bf16_bits(syn.normal_rows(2, 0, int(off[-1]), 256))
    Wg = syn.to_bf16_bits(syn.normal_rows(2, 1, 4 * 256, 256, std=0.02)).reshape(4, 256, 256)
    offd = torch.from_numpy(off).cuda()
    out["grouped"] = digest(bi.grouped_gemm_bf16(dev(Xg), dev(Wg), offd))
    out["grouped_silu"] = digest(bi.grouped_gemm_silu_bf16(dev(Xg), dev(Wg), offd))
    # NVFP4 quantiser and GEMM
    a = syn.to_bf16_bits(syn.normal_rows(3, syn.TID_FP4_A, 130, 1024))
    gs = float(syn.nvfp4_global_scale(syn.bf16_bits_to_f32(a)))
    Q, S = bi.quantize_nvfp4(dev(a), gs)
    out["quantize"] = digest(Q) + digest(S)
    d = syn.nvfp4_inputs(1, 512, 1024, seed=3)
    out["nvfp4"] = digest(bi.gemm_nvfp4(Q, S, torch.from_numpy(d["B"]).cuda(), torch.from_numpy(d["SB_il"]).cuda(), 0.5))
    # RMSNorm with and without residual, and the rank-ordered sum
    x, res, w, _ = syn.rmsnorm_inputs(33, 4096, seed=4)
    rd = dev(res)
    out["rmsnorm_res"] = digest(bi.rmsnorm(dev(x), dev(w), 1e-6, residual=rd)) + digest(rd)
    out["rmsnorm"] = digest(bi.rmsnorm(dev(x), dev(w), 1e-6))
    parts = [dev(syn.to_bf16_bits(syn.normal_rows(5, r, 33, 4096))) for r in range(3)]
    out["rank_sum"] = digest(bi.rank_sum_rmsnorm(parts, dev(w), 1e-6))
    # MoE surroundings
    T, E = 40, 128
    logits = torch.from_numpy(syn.normal_rows(6, syn.TID_LOGITS, T, E)).cuda()
    ids, wts = bi.moe_topk_softmax(logits, 8)
    o2, rt, pos = bi.moe_align(ids, E)
    hidden = dev(syn.to_bf16_bits(syn.normal_rows(6, syn.TID_HIDDEN, T, 2048)))
    Xs = bi.moe_gather(hidden, rt)
    y = dev(syn.to_bf16_bits(syn.normal_rows(7, 0, Xs.shape[0], 2048)))
    out["moe"] = digest(ids) + digest(wts) + digest(o2) + digest(Xs) + digest(bi.moe_combine(y, pos, wts))
    out["silu_mul"] = digest(bi.silu_mul(dev(syn.to_bf16_bits(syn.normal_rows(8, 0, 20, 512)))))
    # decode and extend attention
    Hq, Hkv, D, bs = 32, 8, 128, 16
    lens = np.array([300, 17], np.int32)
    nb = 19
    K = dev(syn.to_bf16_bits(syn.normal_rows(9, 0, 2 * nb * bs, Hkv * D)).reshape(2 * nb, bs, Hkv, D))
    V = dev(syn.to_bf16_bits(syn.normal_rows(9, 1, 2 * nb * bs, Hkv * D)).reshape(2 * nb, bs, Hkv, D))
    table = torch.from_numpy(np.arange(2 * nb, dtype=np.int32)[::-1].copy().reshape(2, nb)).cuda()
    Qd = dev(syn.to_bf16_bits(syn.normal_rows(9, 2, 2 * Hq, D)).reshape(2, Hq, D))
    ld = torch.from_numpy(lens).cuda()
    out["decode"] = digest(bi.attention_decode(Qd, K, V, table, ld, 304, D ** -0.5))
    cu = torch.tensor([0, 40, 57], dtype=torch.int32, device="cuda")
    Qe = dev(syn.to_bf16_bits(syn.normal_rows(9, 3, 57 * Hq, D)).reshape(57, Hq, D))
    out["extend"] = digest(bi.attention_extend(Qe, cu, K, V, table, ld, 304, 40, D ** -0.5))
    torch.cuda.synchronize()
    out["status"] = bi.status_string(bi.device_status())
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
