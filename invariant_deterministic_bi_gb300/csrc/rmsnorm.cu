// rmsnorm.cu -- RMSNorm (+ optional residual add) with a fixed reduction tree.
//
// The fused all-reduce + RMSNorm that vLLM PR #51292 ("Disable
// fuse_allreduce_rms under VLLM_BATCH_INVARIANT") turns off reduces with
// shuffles and block reductions in an order that varies from run to run.
// Here the order is a function of H alone:
//   - one CTA of T threads owns one row (T = 128 for H <= 16384, 512 above);
//     thread t owns the 16-byte vectors t, t+T, t+2T, ... (8 bf16 each) and
//     sums the squares of its elements in index order (fp32 FMA);
//   - each warp combines its 32 thread sums with the xor-shuffle butterfly
//     16, 8, 4, 2, 1 (every lane ends with the same value: fp32 addition
//     commutes);
//   - thread 0 adds the warp sums in warp order through shared memory and
//     broadcasts the total.
// Rows never interact, so a row's output does not depend on M or on which CTA
// processes it.
//
// Memory: 128-bit loads and stores, coalesced (thread t reads bytes 16t ..
// 16t+15 of each 16T-byte segment). With 4 vectors per thread at H = 4096 the
// kernel needs few registers, so 10 to 16 CTAs (40 to 64 warps) fit on an SM
// and every SM keeps 160-256 KB of loads in flight. x and residual are
// streamed (evict-first); the weight row stays cached, and its vectors are
// loaded together with the row's where that pays (launch_one below).
#include <cuda_bf16.h>

#include <atomic>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// h = bf16(x + r) for 8 packed elements.
__device__ __forceinline__ uint4 add_round(uint4 a, uint4 b) {
    uint4 h;
    h.x = pack_bf16x2(__float_as_uint(bf_lo(a.x) + bf_lo(b.x)), __float_as_uint(bf_hi(a.x) + bf_hi(b.x)));
    h.y = pack_bf16x2(__float_as_uint(bf_lo(a.y) + bf_lo(b.y)), __float_as_uint(bf_hi(a.y) + bf_hi(b.y)));
    h.z = pack_bf16x2(__float_as_uint(bf_lo(a.z) + bf_lo(b.z)), __float_as_uint(bf_hi(a.z) + bf_hi(b.z)));
    h.w = pack_bf16x2(__float_as_uint(bf_lo(a.w) + bf_lo(b.w)), __float_as_uint(bf_hi(a.w) + bf_hi(b.w)));
    return h;
}

// ss += h_k^2 for the 8 elements in index order.
__device__ __forceinline__ float sum_squares(uint4 h, float ss) {
    const uint32_t v[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = bf_lo(v[i]), hi = bf_hi(v[i]);
        ss = __fmaf_rn(lo, lo, ss);
        ss = __fmaf_rn(hi, hi, ss);
    }
    return ss;
}

// bf16(h * r * w) for 8 elements.
__device__ __forceinline__ uint4 scale(uint4 h, uint4 w, float r) {
    const uint32_t hv[4] = {h.x, h.y, h.z, h.w}, wv[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __fmul_rn(__fmul_rn(bf_lo(hv[i]), r), bf_lo(wv[i]));
        const float hi = __fmul_rn(__fmul_rn(bf_hi(hv[i]), r), bf_hi(wv[i]));
        o[i] = pack_bf16x2(__float_as_uint(lo), __float_as_uint(hi));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 1 / sqrt(sum/H + eps) for the whole CTA: warp butterflies, then the warp sums
// in warp order. `red` holds T/32 + 1 floats.
template <int T>
__device__ __forceinline__ float row_scale(float ss, int H, float eps, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float total = red[0];
#pragma unroll
        for (int w = 1; w < T / 32; ++w) total += red[w];
        red[T / 32] = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(total, static_cast<float>(H)) + eps));
    }
    __syncthreads();
    return red[T / 32];
}

// One row per CTA; VPT vectors per thread (H <= 8 * T * VPT). WPRE: the
// thread's weight vectors are loaded with the row, so the scaling after the
// reduction waits for no load (VPT more registers a thread); otherwise they
// are loaded after the reduction.
template <int T, int VPT, bool RESIDUAL, bool WPRE>
__global__ void __launch_bounds__(T)
rmsnorm_kernel(const uint4 *x, uint4 *residual, const uint4 *__restrict__ w, uint4 *out, int H, float eps) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ float red[T / 32 + 1];
    const int64_t row = blockIdx.x;
    const int nvec = H >> 3;
    const int t = threadIdx.x;
    const uint4 *xr = x + row * nvec;
    uint4 *rr = RESIDUAL ? residual + row * nvec : nullptr;
    uint4 h[VPT], wv[VPT];
    if (WPRE) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int j = t + T * i;
            if (j < nvec) wv[i] = __ldg(w + j);
        }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int j = t + T * i;
        if (j < nvec) {
            h[i] = __ldcs(xr + j);
            if (RESIDUAL) h[i] = add_round(h[i], __ldcs(rr + j));
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int j = t + T * i;
        if (j < nvec) {
            if (RESIDUAL) __stcs(rr + j, h[i]);
            ss = sum_squares(h[i], ss);
        }
    }
    const float r = row_scale<T>(ss, H, eps, red);
    uint4 *orow = out + row * nvec;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int j = t + T * i;
        if (j < nvec) __stcs(orow + j, scale(h[i], WPRE ? wv[i] : __ldg(w + j), r));
    }
}

// ---- Deterministic tensor-parallel all-reduce + RMSNorm: R ranks' partial
// rows (all readable from this GPU) are summed in rank order 0, 1, ..., R-1 in
// fp32 and rounded once to bf16 (the all-reduced row), then the residual add
// and the RMSNorm above follow with the same tree. vLLM PR #51292 turns off
// its fused all-reduce + RMSNorm under batch invariance because that kernel's
// reduction order varies between runs; here the order is the rank index.
constexpr int kMaxRanks = 16;
// Passed as a __grid_constant__ kernel parameter: p[r] with a run-time r is
// read from parameter space instead of from a per-thread local copy.
struct RankParts {
    const uint4 *p[kMaxRanks];
};

// PRE: the row's residual and weight vectors are loaded before the rank sum
// (2 VPT more registers a thread), so after the sum no load waits; otherwise
// the residual is loaded after the sum and the weights after the reduction.
// UNR: ranks whose loads are in flight together (the rank loop's unrolling).
template <int T, int VPT, bool RESIDUAL, bool PRE, int UNR>
__global__ void __launch_bounds__(T)
rank_sum_rmsnorm_kernel(const __grid_constant__ RankParts parts, int R, uint4 *residual, const uint4 *__restrict__ w, uint4 *sum_out,
                        uint4 *out, int H, float eps) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ float red[T / 32 + 1];
    const int64_t row = blockIdx.x;
    const int nvec = H >> 3;
    const int t = threadIdx.x;
    uint4 *rr = RESIDUAL ? residual + row * nvec : nullptr;
    // Every element is summed over the ranks in order 0, 1, ..., R-1. Up to
    // 8 vectors a thread, the rank loop is outside the row's vectors so that
    // each thread has VPT (twice that, unrolled) independent loads in flight
    // rather than one; longer rows keep one vector's sum at a time.
    uint4 h[VPT], rv[VPT], wv[VPT];
    if (PRE) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int j = t + T * i;
            if (j < nvec) {
                wv[i] = __ldg(w + j);
                if (RESIDUAL) rv[i] = __ldcs(rr + j);
            }
        }
    }
    auto finish = [&](int i, int j, const float (&acc)[8]) {
        uint4 a;
        a.x = pack_bf16x2(__float_as_uint(acc[0]), __float_as_uint(acc[1]));
        a.y = pack_bf16x2(__float_as_uint(acc[2]), __float_as_uint(acc[3]));
        a.z = pack_bf16x2(__float_as_uint(acc[4]), __float_as_uint(acc[5]));
        a.w = pack_bf16x2(__float_as_uint(acc[6]), __float_as_uint(acc[7]));
        if (sum_out) __stcs(sum_out + row * nvec + j, a);
        h[i] = RESIDUAL ? add_round(a, PRE ? rv[i] : __ldcs(rr + j)) : a;
    };
    auto add8 = [](float (&acc)[8], const uint4 &v) {
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc[2 * q] = __fadd_rn(acc[2 * q], bf_lo(vw[q]));
            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf_hi(vw[q]));
        }
    };
    if constexpr (VPT <= 8) {
        float acc[VPT][8];
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
#pragma unroll UNR
        for (int r = 0; r < R; ++r) {
            uint4 v[VPT];
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int j = t + T * i;
                v[i] = j < nvec ? __ldcs(parts.p[r] + row * nvec + j) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < VPT; ++i) add8(acc[i], v[i]);
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int j = t + T * i;
            if (j < nvec) finish(i, j, acc[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int j = t + T * i;
            if (j < nvec) {
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int r = 0; r < R; ++r) add8(acc, __ldcs(parts.p[r] + row * nvec + j));
                finish(i, j, acc);
            }
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int j = t + T * i;
        if (j < nvec) {
            if (RESIDUAL) __stcs(rr + j, h[i]);
            ss = sum_squares(h[i], ss);
        }
    }
    const float r = row_scale<T>(ss, H, eps, red);
    uint4 *orow = out + row * nvec;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int j = t + T * i;
        if (j < nvec) __stcs(orow + j, scale(h[i], PRE ? wv[i] : __ldg(w + j), r));
    }
}

// Threads per row and vectors per thread, chosen from H alone.
struct RowShape {
    int threads, vpt;
};
RowShape row_shape(int64_t H) {
    const int64_t nvec = H / 8;
    if (nvec <= 128 * 16) {
        int vpt = 1;
        while (128 * vpt < nvec) vpt *= 2;
        return {128, vpt};
    }
    int vpt = 1;
    while (512 * vpt < nvec) vpt *= 2;
    return {512, vpt};
}

// Resident CTAs per SM of a kernel launched with T threads, queried once.
template <typename Kernel>
int resident_per_sm(Kernel kernel, int T, std::atomic<int> &cache) {
    int n = cache.load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, T, 0) != cudaSuccess || n < 1) n = 1;
        cache.store(n, std::memory_order_relaxed);
    }
    return n;
}

// Whether M rows take a kernel's early-load form `pre` (more registers, no
// load after the reduction) over its plain form: always while all M rows'
// CTAs fit on the GPU at once, where a row's latency is the time; beyond,
// only when `pre` keeps at least 3/4 of the plain form's CTAs per SM (the
// loads in flight that set the rate), and only if `ratio_ok` allows it.
template <typename Kernel>
bool take_pre(Kernel pre, Kernel plain, int T, int64_t M, bool ratio_ok, std::atomic<int> (&cache)[2]) {
    int dev;
    const DeviceInfo *info;
    if (current_device(&dev, &info) != BI_OK) return false;
    const int np = resident_per_sm(pre, T, cache[0]);
    if (M <= static_cast<int64_t>(np) * info->sm_count) return true;
    return ratio_ok && 4 * np >= 3 * resident_per_sm(plain, T, cache[1]);
}

// RMSNorm: the form with the weight vectors loaded with the row (WPRE) for up
// to 8 vectors a thread; measured at H = 4096 it is faster at every M without
// the residual (48 against 38 registers: 10 against 12 CTAs an SM) and slower
// beyond one wave with it (56 against 32: 9 against 16). Which form runs
// changes no arithmetic.
template <int T, int VPT, bool RES>
bi_status launch_one(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                     cudaStream_t s) {
    auto kernel = rmsnorm_kernel<T, VPT, RES, false>;
    if constexpr (VPT <= 8) {
        static std::atomic<int> cache[2];
        if (take_pre(rmsnorm_kernel<T, VPT, RES, true>, kernel, T, M, true, cache))
            kernel = rmsnorm_kernel<T, VPT, RES, true>;
    }
    return launch_pdl(kernel, dim3(static_cast<unsigned>(M)), dim3(T), 0, s, static_cast<const uint4 *>(x),
                      static_cast<uint4 *>(residual), static_cast<const uint4 *>(w), static_cast<uint4 *>(out),
                      static_cast<int>(H), eps);
}

template <bool RES>
bi_status launch_res(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                     cudaStream_t s) {
    const RowShape rs = row_shape(H);
    if (rs.threads == 128) {
        switch (rs.vpt) {
            case 1: return launch_one<128, 1, RES>(x, residual, w, out, M, H, eps, s);
            case 2: return launch_one<128, 2, RES>(x, residual, w, out, M, H, eps, s);
            case 4: return launch_one<128, 4, RES>(x, residual, w, out, M, H, eps, s);
            case 8: return launch_one<128, 8, RES>(x, residual, w, out, M, H, eps, s);
            default: return launch_one<128, 16, RES>(x, residual, w, out, M, H, eps, s);
        }
    }
    switch (rs.vpt) {
        case 1: return launch_one<512, 1, RES>(x, residual, w, out, M, H, eps, s);
        case 2: return launch_one<512, 2, RES>(x, residual, w, out, M, H, eps, s);
        case 4: return launch_one<512, 4, RES>(x, residual, w, out, M, H, eps, s);
        case 8: return launch_one<512, 8, RES>(x, residual, w, out, M, H, eps, s);
        default: return launch_one<512, 16, RES>(x, residual, w, out, M, H, eps, s);
    }
}

// The rank sum's forms. Large M: the plain form, two ranks' loads in flight.
// While all M rows' CTAs fit on the GPU at once (a row's latency is the time;
// up to 8 vectors a thread): R <= 2 the early-load form (PRE), R = 3..4 PRE
// with four ranks' loads in flight, R > 4 the plain form with four. The same
// operations in the same order either way. Measured at H = 4096 (M = 1 and
// 128): R = 2 3.1 -> 1.75 and 4.0 -> 2.4 us; R = 4 3.85 -> 2.0 and 3.9 ->
// 2.25 us; R = 8 5.1 -> 3.7 and 8.4 -> 5.5 us. Four ranks in flight at
// M = 16384 cost 6-23 % (fewer CTAs an SM), and at R = 2 PRE with four was
// slower than with two (1.97 against 1.75 us).
template <int T, int VPT, bool RES>
bi_status launch_rank_one(const RankParts &parts, int R, void *residual, const void *w, void *sum_out, void *out,
                          int64_t M, int64_t H, float eps, cudaStream_t s) {
    auto kernel = rank_sum_rmsnorm_kernel<T, VPT, RES, false, 2>;
    if constexpr (VPT <= 8) {
        if (R <= 2) {
            static std::atomic<int> cache[2];
            if (take_pre(rank_sum_rmsnorm_kernel<T, VPT, RES, true, 2>, kernel, T, M, false, cache))
                kernel = rank_sum_rmsnorm_kernel<T, VPT, RES, true, 2>;
        } else if (R <= 4) {
            static std::atomic<int> cache[2];
            if (take_pre(rank_sum_rmsnorm_kernel<T, VPT, RES, true, 4>, kernel, T, M, false, cache))
                kernel = rank_sum_rmsnorm_kernel<T, VPT, RES, true, 4>;
        } else {
            static std::atomic<int> cache[2];
            if (take_pre(rank_sum_rmsnorm_kernel<T, VPT, RES, false, 4>, kernel, T, M, false, cache))
                kernel = rank_sum_rmsnorm_kernel<T, VPT, RES, false, 4>;
        }
    }
    return launch_pdl(kernel, dim3(static_cast<unsigned>(M)), dim3(T), 0, s, parts, R, static_cast<uint4 *>(residual),
                      static_cast<const uint4 *>(w), static_cast<uint4 *>(sum_out), static_cast<uint4 *>(out),
                      static_cast<int>(H), eps);
}

template <bool RES>
bi_status launch_rank_res(const RankParts &parts, int R, void *residual, const void *w, void *sum_out, void *out,
                          int64_t M, int64_t H, float eps, cudaStream_t s) {
    const RowShape rs = row_shape(H);
    if (rs.threads == 128) {
        switch (rs.vpt) {
            case 1: return launch_rank_one<128, 1, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
            case 2: return launch_rank_one<128, 2, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
            case 4: return launch_rank_one<128, 4, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
            case 8: return launch_rank_one<128, 8, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
            default: return launch_rank_one<128, 16, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
        }
    }
    switch (rs.vpt) {
        case 1: return launch_rank_one<512, 1, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
        case 2: return launch_rank_one<512, 2, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
        case 4: return launch_rank_one<512, 4, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
        case 8: return launch_rank_one<512, 8, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
        default: return launch_rank_one<512, 16, RES>(parts, R, residual, w, sum_out, out, M, H, eps, s);
    }
}

__global__ void wait_timeout_check_kernel(unsigned *status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, nullptr, limit_ns)) atomicOr(status, kDevTimeout);
}

// One thread writes element `index` of a 64-element array under the debug
// build's bounds check against `limit` (an index >= limit is skipped and recorded).
__device__ unsigned g_bounds_probe[64];
__global__ void bounds_check_kernel(int index, int limit, unsigned *status) {
    if (BI_IN_BOUNDS(index < limit, status)) g_bounds_probe[index & 63] = 1u;
}

}  // namespace

void plan_rmsnorm(int64_t M, int64_t H, bi_plan_t *pl) {
    const RowShape rs = row_shape(H);
    pl->op = BI_OP_RMSNORM;
    pl->block_m = 1;                               // rows per CTA
    pl->block_n = static_cast<int32_t>(H);
    pl->block_k = 8;                               // elements per vector
    pl->mma_m = pl->mma_n = pl->mma_k = 0;
    pl->k_steps = rs.vpt;                          // vectors per thread
    pl->split_k = 1;
    pl->stages = 1;
    pl->threads = rs.threads;
    pl->smem_bytes = static_cast<int32_t>((rs.threads / 32 + 1) * 4);
    pl->tiles_m = M;
    pl->tiles_n = 1;
    pl->grid = static_cast<int32_t>(M);
    pl->reduce_tree = rs.vpt * 8;                  // elements each thread sums in order
}

bi_status launch_rmsnorm(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                         cudaStream_t s) {
    return residual ? launch_res<true>(x, residual, w, out, M, H, eps, s)
                    : launch_res<false>(x, residual, w, out, M, H, eps, s);
}

bi_status launch_rank_sum_rmsnorm(const void *const *parts, int32_t R, void *residual, const void *w, void *sum_out,
                                  void *out, int64_t M, int64_t H, float eps, cudaStream_t s) {
    RankParts rp{};
    for (int r = 0; r < R; ++r) rp.p[r] = static_cast<const uint4 *>(parts[r]);
    return residual ? launch_rank_res<true>(rp, R, residual, w, sum_out, out, M, H, eps, s)
                    : launch_rank_res<false>(rp, R, residual, w, sum_out, out, M, H, eps, s);
}

bi_status launch_bounds_check(int32_t index, int32_t limit, cudaStream_t s) {
    bounds_check_kernel<<<1, 1, 0, s>>>(index, limit, device_status_word());
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

bi_status launch_wait_timeout_check(uint32_t limit_us, cudaStream_t s) {
    wait_timeout_check_kernel<<<1, 32, 0, s>>>(device_status_word(), static_cast<unsigned long long>(limit_us) * 1000ull);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace bi
