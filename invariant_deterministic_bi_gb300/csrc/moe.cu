// moe.cu -- the batch-invariant MoE layer around bi_grouped_gemm_bf16:
// routing (top-k softmax), expert alignment, gather, SiLU-mul and the
// weighted combine, for the MoE models the vllm-ascend "Batch Invariance"
// guide lists as tested (Qwen3-30B-A3B, Qwen3-235B-A22B).
//
// Invariance: routing, gather, SiLU-mul and combine are per token (or per
// row) with fixed reduction orders; the alignment only decides *where* a
// token's rows sit, never their values; the combine adds a token's k expert
// outputs in top-k rank order. So a token's layer output does not depend on
// which tokens share the batch. No atomics anywhere (the alignment uses
// per-expert block scans), so every buffer is the same bits run to run.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// --------------------------------------------------------------- routing
// One warp per token. Lane l holds logits l, l+32, ...; max and the sum of
// exponentials use fixed per-lane orders and xor butterflies; the k winners
// come from k warp arg-max rounds under the total order (larger logit, then
// lower expert index), each round two warp reductions (redux.sync) on
// order-preserving integer keys.
template <int MAXJ>
__global__ void __launch_bounds__(256)
topk_softmax_kernel(const float *__restrict__ logits, int64_t T, int E, int k, int renorm, int32_t *__restrict__ ids,
                    float *__restrict__ wout) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + warp;
    if (t >= T) return;                       // whole warp leaves together
    const float *l = logits + t * E;
    float v[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? l[e] : -INFINITY;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) mx = fmaxf(mx, v[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j)
        if (lane + 32 * j < E) s += expf(v[j] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);

    // each round: the lane's best untaken logit as an order-preserving key
    // (zero of either sign as +0, so equal logits stay equal), the warp's
    // largest key by one reduction, then the lowest expert holding it
    uint32_t kv[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
        const uint32_t u = __float_as_uint(v[j] == 0.0f ? 0.0f : v[j]);
        kv[j] = lane + 32 * j < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;   // 0: no expert
    }
    float my_v = 0.0f;                         // lane i < k: the logit of rank i
    int32_t my_id = 0;                         // lane i < k: the expert of rank i
    for (int i = 0; i < k; ++i) {
        uint32_t lk = 0u, le = 0x7fffffffu;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
            if (kv[j] > lk) {                  // strict: the lane's lower expert wins a tie
                lk = kv[j];
                le = lane + 32 * j;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, lk);
        const uint32_t be = __reduce_min_sync(0xffffffffu, lk == mk ? le : 0x7fffffffu);
        if ((be & 31u) == static_cast<uint32_t>(lane)) {
#pragma unroll
            for (int j = 0; j < MAXJ; ++j)
                if (j == static_cast<int>(be >> 5)) kv[j] = 0u;   // taken
        }
        if (lane == i) {
            my_v = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
            my_id = static_cast<int32_t>(be);
        }
    }
    // rank i's weight e^(v - max) / sum on lane i, then the weights' sum in
    // rank order 0, 1, ..., k-1 (every lane adds the same values in turn)
    const float my_w = lane < k ? __fdiv_rn(expf(my_v - mx), s) : 0.0f;
    float wsum = 0.0f;
    for (int i = 0; i < k; ++i) wsum += __shfl_sync(0xffffffffu, my_w, i);
    if (lane < k) {
        ids[t * k + lane] = my_id;
        wout[t * k + lane] = renorm ? __fdiv_rn(my_w, wsum) : my_w;
    }
}

// ------------------------------------------------------------- alignment
// The (token, rank) pairs are cut into S segments of consecutive pairs.
// Step 0 (one block per (expert, segment)): count the segment's pairs routed
// to the expert; the counts go to row_token[e * S + s] (row_token is written
// for real only in step 3, and E * S <= T * k is kept).
// Step 1 (one block per (expert, segment)): give each of the segment's pairs
// routed to the expert its rank among all of the expert's pairs: the counts
// of the expert's earlier segments plus its rank inside the segment. Each
// pass covers 1024 pairs: thread t holds pairs 4t..4t+3 of the pass, an
// inclusive shuffle scan gives the thread's offset in its warp, and the warp
// totals are added in warp order. The last segment's block writes the
// expert's count to offsets[e + 1]. All integer: the result is the unique
// stable order, whatever the segmentation.
__device__ __forceinline__ void match4(const int32_t *ids, int64_t p0, int64_t end, int e, bool vec_ok, int (&f)[4]) {
    if (vec_ok && p0 + 3 < end) {
        const int4 v = *reinterpret_cast<const int4 *>(ids + p0);
        f[0] = v.x == e; f[1] = v.y == e; f[2] = v.z == e; f[3] = v.w == e;
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) f[q] = (p0 + q < end) && ids[p0 + q] == e;
    }
}

__global__ void __launch_bounds__(256)
align_count_kernel(const int32_t *__restrict__ ids, int64_t P, int64_t seg, int S, int32_t *__restrict__ counts) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ int warp_tot[8];
    const int e = blockIdx.x / S, sgi = blockIdx.x - e * S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15u) == 0;   // 16-byte loads only when aligned
    const int64_t begin = sgi * seg, end = min(P, begin + seg);
    int c = 0;
    for (int64_t p0 = begin + 4 * static_cast<int64_t>(threadIdx.x); p0 < end; p0 += 1024) {
        int f[4];
        match4(ids, p0, end, e, vec_ok, f);
        c += f[0] + f[1] + f[2] + f[3];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) warp_tot[warp] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += warp_tot[w];
        counts[e * S + sgi] = tot;
    }
}

__global__ void __launch_bounds__(256)
align_rank_kernel(const int32_t *__restrict__ ids, int64_t P, int64_t seg, int S, const int32_t *__restrict__ counts,
                  int32_t *__restrict__ pos, int32_t *__restrict__ offsets) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ int warp_tot[8];
    const int e = blockIdx.x / S, sgi = blockIdx.x - e * S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ids) & 15u) == 0;
    const int64_t begin = sgi * seg, end = min(P, begin + seg);
    int running = 0;
    for (int i = 0; i < sgi; ++i) running += counts[e * S + i];       // the expert's earlier segments
    for (int64_t base = begin; base < end; base += 1024) {
        const int64_t p0 = base + 4 * static_cast<int64_t>(threadIdx.x);
        int f[4];
        match4(ids, p0, end, e, vec_ok, f);
        const int cnt = f[0] + f[1] + f[2] + f[3];
        int incl = cnt;                                   // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int before = 0, chunk = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            before += w < warp ? warp_tot[w] : 0;
            chunk += warp_tot[w];
        }
        int r = running + before + incl - cnt;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (f[q]) pos[p0 + q] = r++;
        running += chunk;
        __syncthreads();
    }
    if (threadIdx.x == 0 && sgi == S - 1) {
        offsets[e + 1] = running;
        if (e == 0) offsets[0] = 0;
    }
}

// Few pairs (at most kSmallAlign): the whole alignment in one block. The ids
// are staged in shared memory by all threads; warp 0 walks the pairs in
// order, 32 at a time: the lanes routed to the same
// expert are grouped (__match_any_sync), a pair's rank is the expert's
// running count plus the lanes before it in its group, and the group's
// lowest lane advances the count. Then the counts are scanned into offsets
// and every thread places its pairs. Integer only: the same unique stable
// order as the multi-block path.
constexpr int kSmallAlign = 128;

// Inclusive prefix sum of one int per thread over a block of 1024 threads:
// shuffle scans inside each warp, then over the 32 warp totals (integer adds,
// so the order does not matter). `wsum` holds 32 ints.
__device__ __forceinline__ int block_inclusive_scan_1024(int v, int *wsum) {
    const int t = threadIdx.x, lane = t & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) wsum[t >> 5] = v;
    __syncthreads();
    if (t < 32) {
        int w = wsum[t];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[t] = w;
    }
    __syncthreads();
    return t >= 32 ? v + wsum[(t >> 5) - 1] : v;
}

__global__ void __launch_bounds__(1024)
align_small_kernel(const int32_t *__restrict__ ids, int P, int k, int E, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ row_token, int32_t *__restrict__ pos, unsigned *status) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ int cnt[1024];                 // per expert: pairs so far, then all its pairs
    __shared__ int incl[1024];                // inclusive prefix of the counts
    __shared__ int rank[kSmallAlign];         // a pair's rank within its expert; -1: id outside [0, E)
    __shared__ int id_s[kSmallAlign];
    const int t = threadIdx.x, lane = t & 31;
    cnt[t] = 0;
    for (int p = t; p < P; p += 1024) id_s[p] = ids[p];
    __syncthreads();
    if (t < 32) {
        bool bad = false;
        for (int p0 = 0; p0 < P; p0 += 32) {
            const int p = p0 + lane;
            int e = p < P ? id_s[p] : -1;
            if (p < P && (e < 0 || e >= E)) {
                bad = true;
                e = -1;
            }
            const unsigned same = __match_any_sync(0xffffffffu, e);
            const int before = __popc(same & ((1u << lane) - 1u));
            const int base = e >= 0 ? cnt[e] : 0;
            __syncwarp();
            if (p < P) rank[p] = e >= 0 ? base + before : -1;
            if (e >= 0 && before == 0) cnt[e] = base + __popc(same);
            __syncwarp();
        }
        if (bad) atomicOr(status, kDevBadOffsets);
    }
    __syncthreads();
    __shared__ int wsum[32];
    incl[t] = block_inclusive_scan_1024(t < E ? cnt[t] : 0, wsum);
    __syncthreads();
    if (t < E) offsets[t + 1] = incl[t];
    if (t == 0) offsets[0] = 0;
    for (int p = t; p < P; p += 1024) {
        const int r = rank[p];
        if (r < 0) continue;
        const int e = id_s[p];
        const int o = incl[e] - cnt[e] + r;
        pos[p] = o;
        row_token[o] = p / k;
    }
}

// Step 2 (one block): offsets[1..E] counts -> inclusive prefix, in place.
__global__ void __launch_bounds__(1024) align_scan_kernel(int32_t *offsets, int E) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    __shared__ int wsum[32];
    const int i = threadIdx.x;
    const int v = block_inclusive_scan_1024(i < E ? offsets[i + 1] : 0, wsum);
    if (i < E) offsets[i + 1] = v;
}

// Step 3: pos = offsets[expert] + rank; row_token[pos] = token.
__global__ void __launch_bounds__(256)
align_scatter_kernel(const int32_t *__restrict__ ids, int64_t P, int k, int E, const int32_t *__restrict__ offsets,
                     int32_t *__restrict__ pos, int32_t *__restrict__ row_token, unsigned *status) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; p < P;
         p += static_cast<int64_t>(gridDim.x) * 256) {
        const int e = ids[p];
        if (e < 0 || e >= E) {
            atomicOr(status, kDevBadOffsets);
            continue;
        }
        const int r = offsets[e] + pos[p];
        pos[p] = r;
        row_token[r] = static_cast<int32_t>(p / k);
    }
}

// ----------------------------------------------------------------- gather
// One warp per destination row at a time (grid-stride over rows): the source
// token index is read once, and each lane moves up to 8 of the row's 16-byte
// pieces with all its loads in flight before its stores, which are streaming
// stores (55.6 -> 49.7 us at 65536 rows of 4 KB: the sorted copy is read once,
// by the expert GEMM, and need not displace the token rows in L2).
__global__ void __launch_bounds__(256)
gather_kernel(const uint4 *__restrict__ hidden, int64_t T, int64_t hv, const int32_t *__restrict__ row_token,
              int64_t rows, uint4 *__restrict__ out, unsigned *status) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    constexpr int kPer = 8;
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * 8;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
        const int64_t t = row_token[r];
        if (t < 0 || t >= T) {
            if (lane == 0) atomicOr(status, kDevBadOffsets);
            continue;
        }
        const uint4 *src = hidden + t * hv;
        uint4 *dst = out + r * hv;
        for (int64_t j0 = lane; j0 < hv; j0 += 32 * kPer) {
            uint4 v[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u)
                if (j0 + 32 * u < hv) v[u] = __ldg(src + j0 + 32 * u);
#pragma unroll
            for (int u = 0; u < kPer; ++u)
                if (j0 + 32 * u < hv) __stcs(dst + j0 + 32 * u, v[u]);   // streamed: read once, later
        }
    }
}

// --------------------------------------------------------------- SiLU-mul
// act = bf16( silu(g) * u ), silu(g) = g / (1 + exp(-g)), fp32 (silu_mul_f32); rows are [gate | up].
__global__ void __launch_bounds__(256)
silu_mul_kernel(const uint4 *__restrict__ gu, int64_t rows, int64_t iv, uint4 *__restrict__ act) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    const int64_t total = rows * iv;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * 256) {
        const int64_t r = i / iv, j = i - r * iv;
        const uint4 g = __ldcs(gu + r * 2 * iv + j), u = __ldcs(gu + r * 2 * iv + iv + j);
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float g0 = bf_lo(gw[q]), g1 = bf_hi(gw[q]);
            const float a0 = silu_mul_f32(g0, bf_lo(uw[q]));
            const float a1 = silu_mul_f32(g1, bf_hi(uw[q]));
            o[q] = pack_bf16x2(__float_as_uint(a0), __float_as_uint(a1));
        }
        __stcs(act + i, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

// ---------------------------------------------------------------- combine
// out[t] = bf16( sum_{i = 0..k-1} w[t][i] * Y[pos[t][i]] ), fp32 FMA in rank order.
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ Y, int64_t rows, const int32_t *__restrict__ pos,
               const float *__restrict__ w, int k, int64_t hv, uint4 *__restrict__ out, unsigned *status) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    const int64_t t = blockIdx.x;
    for (int64_t j = threadIdx.x; j < hv; j += 256) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        bool bad = false;
        for (int i0 = 0; i0 < k; i0 += 8) {          // up to 8 rows' loads in flight, then the FMAs in rank order
            uint4 y[8];
            float wi[8];
            bool ok[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                ok[u] = false;
                if (i0 + u < k) {
                    const int64_t r = pos[t * k + i0 + u];
                    if (r < 0 || r >= rows) {
                        bad = true;
                    } else {
                        wi[u] = w[t * k + i0 + u];
                        y[u] = __ldg(Y + r * hv + j);
                        ok[u] = true;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (!ok[u]) continue;
                const uint32_t yw[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] = __fmaf_rn(wi[u], bf_lo(yw[q]), acc[2 * q]);
                    acc[2 * q + 1] = __fmaf_rn(wi[u], bf_hi(yw[q]), acc[2 * q + 1]);
                }
            }
        }
        if (bad) atomicOr(status, kDevBadOffsets);
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(__float_as_uint(acc[2 * q]), __float_as_uint(acc[2 * q + 1]));
        __stcs(out + t * hv + j, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

inline unsigned grid_for(int64_t items, const DeviceInfo *info) {
    const int64_t g = (items + 255) / 256, cap = static_cast<int64_t>(info->sm_count) * 16;
    return static_cast<unsigned>(g < 1 ? 1 : (g < cap ? g : cap));
}

}  // namespace

bi_status launch_moe_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t k, int32_t renorm, int32_t *ids,
                                  float *w, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((T + 7) / 8));
    auto go = [&](auto kernel) { return launch_pdl(kernel, grid, dim3(256), 0, s, logits, T, E, k, renorm, ids, w); };
    if (E <= 32) return go(topk_softmax_kernel<1>);
    if (E <= 64) return go(topk_softmax_kernel<2>);
    if (E <= 128) return go(topk_softmax_kernel<4>);
    if (E <= 256) return go(topk_softmax_kernel<8>);
    if (E <= 512) return go(topk_softmax_kernel<16>);
    return go(topk_softmax_kernel<32>);
}

bi_status launch_moe_align(const int32_t *ids, int64_t T, int32_t k, int32_t E, int32_t *offsets, int32_t *row_token,
                           int32_t *pos, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    const int64_t P = T * k;
    if (P <= kSmallAlign)
        return launch_pdl(align_small_kernel, dim3(1), dim3(1024), 0, s, ids, static_cast<int>(P), k, E, offsets,
                          row_token, pos, device_status_word());
    // segments of whole 1024-pair passes, at most 32 per expert, E * S <= P;
    // below 16384 pairs one segment (no counting pass) is quicker
    int S = 1;
    while (P >= 16384 && S < 32 && static_cast<int64_t>(E) * (2 * S) <= P && P / (2 * S) >= 1024) S *= 2;
    const int64_t seg = ((P + S - 1) / S + 1023) / 1024 * 1024;   // whole passes: 16-byte aligned pair groups
    const dim3 blocks(static_cast<unsigned>(E * S));
    if (S > 1 && (st = launch_pdl(align_count_kernel, blocks, dim3(256), 0, s, ids, P, seg, S, row_token)) != BI_OK)
        return st;
    if ((st = launch_pdl(align_rank_kernel, blocks, dim3(256), 0, s, ids, P, seg, S, row_token, pos, offsets)) != BI_OK)
        return st;
    if ((st = launch_pdl(align_scan_kernel, dim3(1), dim3(1024), 0, s, offsets, E)) != BI_OK) return st;
    return launch_pdl(align_scatter_kernel, dim3(grid_for(P, info)), dim3(256), 0, s, ids, P, k, E, offsets, pos,
                      row_token, device_status_word());
}

bi_status launch_moe_gather(const void *hidden, int64_t T, int64_t H, const int32_t *row_token, int64_t rows,
                            void *out, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    return launch_pdl(gather_kernel, dim3(grid_for(rows * 32, info)), dim3(256), 0, s,
                      static_cast<const uint4 *>(hidden), T, H / 8, row_token, rows, static_cast<uint4 *>(out),
                      device_status_word());
}

bi_status launch_silu_mul(const void *gate_up, int64_t rows, int64_t I, void *act, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    return launch_pdl(silu_mul_kernel, dim3(grid_for(rows * (I / 8), info)), dim3(256), 0, s,
                      static_cast<const uint4 *>(gate_up), rows, I / 8, static_cast<uint4 *>(act));
}

bi_status launch_moe_combine(const void *Y, int64_t rows, const int32_t *pos, const float *w, int64_t T, int32_t k,
                             int64_t H, void *out, cudaStream_t s) {
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(T)), dim3(256), 0, s, static_cast<const uint4 *>(Y),
                      rows, pos, w, k, H / 8, static_cast<uint4 *>(out), device_status_word());
}

}  // namespace bi
