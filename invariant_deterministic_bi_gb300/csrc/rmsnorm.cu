// rmsnorm.cu -- RMSNorm (+ optional residual add) with a fixed reduction tree.
//
// The fused all-reduce + RMSNorm that vLLM PR #51292 ("Disable
// fuse_allreduce_rms under VLLM_BATCH_INVARIANT") turns off reduces with
// shuffles and block reductions in an order that varies from run to run.
// Here the order is a function of H alone:
//   - one warp owns one row; lane l owns the 16-byte vectors l, l+32, l+64, ...
//     (8 bf16 each) and sums the squares of its elements in index order (fp32);
//   - the 32 lane sums are combined by the xor-shuffle butterfly 16, 8, 4, 2, 1,
//     which leaves the same total in every lane (fp32 addition commutes).
// Rows never interact, so a row's output does not depend on M or on which
// warp or CTA processes it.
//
// Memory: 128-bit loads and stores, coalesced across the warp (lane l reads
// bytes 16l .. 16l+15 of each 512-byte segment); x and residual are streamed
// (evict-first), the weight row stays cached. For H <= 8192 the row lives in
// registers between the two passes; larger H re-reads it.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kRowsPerCta = 8;   // 8 warps, one row each
constexpr int kThreads = 32 * kRowsPerCta;

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

__device__ __forceinline__ float row_scale(float ss, int H, float eps) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, static_cast<float>(H)) + eps));
}

// Row held in registers: VPL vectors per lane (H <= 256 * VPL).
template <int VPL, bool RESIDUAL>
__global__ void __launch_bounds__(kThreads)
rmsnorm_reg_kernel(const uint4 *x, uint4 *residual, const uint4 *__restrict__ w, uint4 *out, int64_t M,
                   int H, float eps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = H >> 3;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp; row < M;
         row += static_cast<int64_t>(gridDim.x) * kRowsPerCta) {
        const uint4 *xr = x + row * nvec;
        uint4 *rr = RESIDUAL ? residual + row * nvec : nullptr;
        uint4 h[VPL];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            if (j < nvec) {
                h[i] = __ldcs(xr + j);
                if (RESIDUAL) h[i] = add_round(h[i], __ldcs(rr + j));
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            if (j < nvec) {
                if (RESIDUAL) __stcs(rr + j, h[i]);
                ss = sum_squares(h[i], ss);
            }
        }
        const float r = row_scale(ss, H, eps);
        uint4 *orow = out + row * nvec;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            if (j < nvec) __stcs(orow + j, scale(h[i], __ldg(w + j), r));
        }
    }
}

// Any H: the first pass stores h (to residual) and sums; the second re-reads h.
template <bool RESIDUAL>
__global__ void __launch_bounds__(kThreads)
rmsnorm_loop_kernel(const uint4 *x, uint4 *residual, const uint4 *__restrict__ w, uint4 *out, int64_t M, int H,
                    float eps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = H >> 3;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp; row < M;
         row += static_cast<int64_t>(gridDim.x) * kRowsPerCta) {
        const uint4 *xr = x + row * nvec;
        uint4 *rr = RESIDUAL ? residual + row * nvec : nullptr;
        float ss = 0.0f;
        for (int j = lane; j < nvec; j += 32) {
            uint4 h = xr[j];
            if (RESIDUAL) {
                h = add_round(h, rr[j]);
                rr[j] = h;
            }
            ss = sum_squares(h, ss);
        }
        const float r = row_scale(ss, H, eps);
        const uint4 *hr = RESIDUAL ? rr : xr;
        uint4 *orow = out + row * nvec;
        for (int j = lane; j < nvec; j += 32) orow[j] = scale(hr[j], __ldg(w + j), r);
    }
}

template <bool RES>
bi_status launch_res(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                     int grid, cudaStream_t s) {
    auto X = static_cast<const uint4 *>(x);
    auto R = static_cast<uint4 *>(residual);
    auto Wt = static_cast<const uint4 *>(w);
    auto O = static_cast<uint4 *>(out);
    const int h = static_cast<int>(H);
    if (H <= 256) rmsnorm_reg_kernel<1, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else if (H <= 512) rmsnorm_reg_kernel<2, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else if (H <= 1024) rmsnorm_reg_kernel<4, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else if (H <= 2048) rmsnorm_reg_kernel<8, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else if (H <= 4096) rmsnorm_reg_kernel<16, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else if (H <= 8192) rmsnorm_reg_kernel<32, RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    else rmsnorm_loop_kernel<RES><<<grid, kThreads, 0, s>>>(X, R, Wt, O, M, h, eps);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
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

}  // namespace

void plan_rmsnorm(int64_t M, int64_t H, bi_plan_t *pl) {
    pl->op = BI_OP_RMSNORM;
    pl->block_m = kRowsPerCta;
    pl->block_n = static_cast<int32_t>(H);
    pl->block_k = 8;
    pl->mma_m = pl->mma_n = pl->mma_k = 0;
    pl->k_steps = static_cast<int32_t>((H / 8 + 31) / 32);
    pl->split_k = 1;
    pl->stages = 1;
    pl->threads = kThreads;
    pl->smem_bytes = 0;
    pl->tiles_m = (M + kRowsPerCta - 1) / kRowsPerCta;
    pl->tiles_n = 1;
    const int64_t max_grid = 1 << 20;
    pl->grid = static_cast<int32_t>(pl->tiles_m < max_grid ? pl->tiles_m : max_grid);
    pl->reduce_tree = static_cast<int32_t>(((H / 8 + 31) / 32) * 8);
}

bi_status launch_rmsnorm(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                         cudaStream_t s) {
    bi_plan_t pl;
    plan_rmsnorm(M, H, &pl);
    return residual ? launch_res<true>(x, residual, w, out, M, H, eps, pl.grid, s)
                    : launch_res<false>(x, residual, w, out, M, H, eps, pl.grid, s);
}

bi_status launch_wait_timeout_check(uint32_t limit_us, cudaStream_t s) {
    wait_timeout_check_kernel<<<1, 32, 0, s>>>(device_status_word(), static_cast<unsigned long long>(limit_us) * 1000ull);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace bi
