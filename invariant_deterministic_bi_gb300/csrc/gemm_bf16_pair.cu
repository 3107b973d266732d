// gemm_bf16_pair.cu -- batch-invariant bf16 linear layers on CTA pairs (tcgen05 cta_group::2)
// with one K segment: the dense layer Y = X W^T when its plan has one segment
// (the plan and the segmented form are in gemm_bf16_dense.cu), and the
// MoE-grouped layer (for each expert e with rows [off[e], off[e+1]) of the
// expert-sorted X: Y_rows = X_rows W[e]^T, also with SiLU-mul fused).
// This kernel holds no running sum: 192 threads of about 100 registers, so
// under programmatic dependent launch its CTAs can take an SM while the
// previous kernel's last CTAs (an RMSNorm, say) are still finishing there.
//
// 256 x 256 output tiles, each computed by a cluster of two CTAs on two SMs:
//   - each CTA's warp 0 TMA-loads its own 128 rows of the A tile and its own
//     half (128 rows) of the B tile per 64-wide K step into a 6-stage ring;
//     both CTAs' copies complete on the even (leader) CTA's "full" barrier;
//   - one thread of the leader issues tcgen05.mma.cta_group::2 (256 x 256 x 16):
//     the tensor cores of both SMs read A rows from their own CTA and the two
//     B halves from both, and each CTA's 128 accumulator rows land in its own
//     tensor memory (two accumulators of 256 columns, so the epilogue of one
//     tile overlaps the main loop of the next);
//   - the leader's commits are multicast to both CTAs' barriers (stage free,
//     accumulator ready); both CTAs' epilogue warps read their own rows,
//     report back to the leader's "accumulator empty" barrier, and write
//     32 x 64 output boxes through two swizzled 4 KB staging buffers per warp
//     with TMA stores (whole 128-byte lines instead of 16-byte pieces).
// Against the single-CTA 128 x 256 tile this halves the B bytes each SM loads
// and reads from shared memory per MMA (64 instead of 96 bytes per clock at
// full rate) and cuts L2-to-SM traffic per output by a third.
//
// Grouped: a tile never spans two experts -- each expert's rows are cut into
// 256-row tiles of their own (the last one partial), experts in order, M-tiles
// fastest inside an expert so that pairs working at the same time share the
// expert's weight panel in L2; the tile map is built on the device from the
// offsets (prefix of tile counts in shared memory + binary search), with no
// host synchronisation. An epilogue warp whose 32 rows all belong to the
// expert stores them by TMA; one straddling the expert's last row stores the
// rows that exist with 16-byte stores (rows past it belong to the next expert).
//
// Batch invariance: the tile shape, MMA instruction and K order (64-wide K
// steps, four 16-wide MMA steps each, ascending, from zero) are the same for
// every M and every routing, and the same in both modes; rows never interact;
// only which pair computes which tile depends on M (or on the routing).
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kBM = 256;       // pair tile rows (128 per CTA)
constexpr int kHalf = 128;     // rows per CTA of A, and of B
constexpr int kBN = 256;       // pair tile columns = MMA N
constexpr int kBK = 64;
constexpr int kMmaK = 16;
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kGroupM = 8;     // 8 pair tiles (2048 rows) per raster band
constexpr int kABytes = kHalf * kBK * 2;
constexpr int kBBytes = kHalf * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kOutCols = 64;                    // bf16 columns per output box (128 bytes)
constexpr int kOutBytes = 32 * kOutCols * 2;    // one 32-row box
constexpr int kEpiWarps = 4;
constexpr int kBarBytes = 256;
constexpr int kMaxExperts = 1024;
constexpr int kSchedBytes = 2 * (kMaxExperts + 1) * 4;
// Modes of the kernel: the dense layer, the grouped layer, and the grouped
// gate_up layer with SiLU-mul applied in the epilogue.
constexpr int kDense = 0, kGrouped = 1, kGroupedSilu = 2;
// dense: two staging boxes per epilogue warp; grouped: one, plus the tile map
template <int MODE>
__host__ __device__ constexpr int out_boxes() { return MODE == kDense ? 2 : 1; }
template <int MODE>
__host__ __device__ constexpr int smem_bytes() {
    return 1024 + kStages * kStageBytes + kEpiWarps * out_boxes<MODE>() * kOutBytes + kBarBytes +
           (MODE != kDense ? kSchedBytes : 0);
}
static_assert(smem_bytes<kGrouped>() <= 232448 && smem_bytes<kDense>() <= 232448, "shared memory per CTA");

// act = bf16(silu(g) * u) on bf16 g and u: the arithmetic of bi_silu_mul
// (silu_mul_f32), so the fused layer gives the same bits.
__device__ __forceinline__ uint32_t silu_mul_bf16x2(uint32_t g2, uint32_t u2) {
    const float g0 = __uint_as_float(g2 << 16), g1 = __uint_as_float(g2 & 0xFFFF0000u);
    const float u0 = __uint_as_float(u2 << 16), u1 = __uint_as_float(u2 & 0xFFFF0000u);
    return pack_bf16x2(__float_as_uint(silu_mul_f32(g0, u0)), __float_as_uint(silu_mul_f32(g1, u1)));
}
constexpr int kTmemCols = 512;

struct Params {
    int32_t M, N, K;           // dense: M rows; grouped: M = offsets[E] (all rows)
    int32_t a_bytes;           // A bytes each CTA loads per K step (fewer rows when M < 128)
    const int32_t *offsets;    // grouped: device offsets [E+1]
    int32_t E;                 // grouped: experts
    uint8_t *Yg;               // grouped: Y (dense N-strided rows), for rows stored without TMA
    unsigned *status;
};

struct Tile {
    int32_t a_row;     // first row of the pair's 256-row A tile
    int32_t row_end;   // rows >= row_end are not stored
    int32_t n0;        // first output column
    int32_t b_row;     // first row of the pair's 256-row B tile
};

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmY, const Params p) {
    constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN);
    constexpr bool GROUPED = MODE != kDense;
    constexpr bool SILU = MODE == kGroupedSilu;
    // SILU: a tile's 256 accumulator columns are 128 gate columns (B rows from
    // the first half of the expert's weight) and the matching 128 up columns
    // (B rows from the second half); it yields 128 output columns.
    constexpr int kOutTile = SILU ? kBN / 2 : kBN;
    constexpr int kBoxes = out_boxes<MODE>();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    uint8_t *out_stage = smem + kStages * kStageBytes;   // kBoxes staging boxes per epilogue warp
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kEpiWarps * kBoxes * kOutBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *total_s = reinterpret_cast<int *>(tmem_slot + 2);
    int *off_s = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(full) + kBarBytes);   // grouped only
    int *pre_s = off_s + (kMaxExperts + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0: leader (issues the MMAs)
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
    const int num_m = (p.M + kBM - 1) / kBM;
    const int num_n = (p.N + kOutTile - 1) / kOutTile;
    const int k_steps = (p.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);   // 4 epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    grid_dep_wait();      // the set-up above overlaps the previous kernel; global memory only from here
    if constexpr (GROUPED) {
        for (int i = threadIdx.x; i <= p.E; i += kThreads) off_s[i] = p.offsets[i];
        __syncthreads();
        if (warp == 2) {
            // Row-tile prefix over the experts: lane l takes a contiguous block
            // of experts, the block sums are scanned across the warp.
            const int per = (p.E + 31) >> 5;
            const int lo = min(lane * per, p.E), hi = min(lo + per, p.E);
            auto tiles_of = [&](int e) {
                const long long c = static_cast<long long>(off_s[e + 1]) - off_s[e];
                return c > 0 ? static_cast<int>((c + kBM - 1) / kBM) : 0;
            };
            bool ok = true;
            int sum = 0;
            for (int e = lo; e < hi; ++e) {
                if (off_s[e + 1] < off_s[e]) ok = false;
                sum += tiles_of(e);
            }
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            ok = __all_sync(0xffffffffu, ok) && off_s[0] == 0 && off_s[p.E] == p.M;
            int acc = incl - sum;
            for (int e = lo; e < hi; ++e) {
                acc += tiles_of(e);
                pre_s[e + 1] = acc;
            }
            if (lane == 0) pre_s[0] = 0;
            if (lane == 31) *total_s = ok ? incl * num_n : 0;
            if (lane == 0 && !ok && blockIdx.x == 0) atomicOr(p.status, kDevBadOffsets);
        }
    } else {
        if (threadIdx.x == 0) *total_s = num_m * num_n;
    }
    tc_fence_before();
    cluster_sync();                      // both CTAs' barriers exist, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *total_s;

    auto tile_of = [&](int t) -> Tile {
        if constexpr (GROUPED) {
            const int x = t / num_n;
            int lo = 0, hi = p.E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (pre_s[mid] <= x) lo = mid; else hi = mid - 1;
            }
            const int e = lo;
            (void)BI_IN_BOUNDS(e >= 0 && e < p.E && x >= pre_s[e] && x < pre_s[e + 1], p.status);
            const int mt = pre_s[e + 1] - pre_s[e];
            const int local = t - pre_s[e] * num_n;
            const int mb = local % mt, nb = local / mt;
            if constexpr (SILU)   // gate rows [nb*128, +128) of W[e] in CTA 0, up rows [N + nb*128, +128) in CTA 1
                return Tile{off_s[e] + mb * kBM, off_s[e + 1], nb * kOutTile, 2 * e * p.N + nb * kOutTile};
            else
                return Tile{off_s[e] + mb * kBM, off_s[e + 1], nb * kBN, e * p.N + nb * kBN};
        } else {
            const int per_group = kGroupM * num_n;
            const int g = t / per_group;
            const int first = g * kGroupM;
            const int gm = min(kGroupM, num_m - first);
            const int local = t - g * per_group;
            const int mb = first + local % gm, nb = local / gm;
            return Tile{mb * kBM, p.M, nb * kBN, nb * kBN};
        }
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                const Tile tl = tile_of(t);
                const int a_row = tl.a_row + static_cast<int>(rank) * kHalf;
                const int b_row = tl.b_row + static_cast<int>(rank) * (SILU ? p.N : kHalf);
                for (int kb = 0; kb < k_steps; ++kb) {
                    // debug build: the copy's coordinates lie inside the operands (padded to whole tiles)
                    if (!BI_IN_BOUNDS(kb * kBK < p.K && a_row >= 0 && a_row < num_m * kBM + (GROUPED ? p.E * kBM : 0) &&
                                          b_row >= 0, p.status)) { ok = false; break; }
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (p.a_bytes + kBBytes));
                    const uint32_t bar = full_leader + stage * 8;
                    tma_load_2d_pair_bar(sA + stage * kABytes, &tmA, bar, kb * kBK, a_row);
                    tma_load_2d_pair_bar(sB + stage * kBBytes, &tmB, bar, kb * kBK, b_row);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            for (int i = 0; i < kStages && ok; ++i) {   // every stage released by the MMAs
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) ok = false;
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                // The leader's full barriers count both CTAs' bytes: waiting on
                // them lets every copy of the pair in flight land.
                if (rank == 0)
                    for (int s = 0; s < kStages; ++s)
                        if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_phase >> s) & 1u, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (lane == 0 && rank == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < k_steps; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / kMmaK; ++k)
                        mma_bf16_pair(d, sdesc_k_sw128(a0 + k * kMmaK * 2), sdesc_k_sw128(b0 + k * kMmaK * 2), kIdesc,
                                      (kb | k) != 0);
                    tc_commit_pair(&empty[stage], 0x3);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(&tfull[acc], 0x3);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                tc_commit_pair(drain, 0x1);
                mbar_wait(drain, 0, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        // Warp q owns accumulator rows 32q .. 32q+31 of its CTA. Per 64-column
        // box: two 32-column TMEM loads, bf16 rounding, then the box goes into
        // one of the warp's staging buffers (128-byte swizzle: 16-byte chunk c
        // of row r at chunk c ^ (r % 8)) and out by TMA; rows past M and
        // columns past N are clipped by the tensor map. Grouped: a warp whose
        // rows cross the end of the expert stores its rows that exist directly.
        const int q = warp & 3;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        uint8_t *boxes = out_stage + q * kBoxes * kOutBytes;
        if (lane == 0) tma_prefetch_desc(&tmY);
        int it = 0;
        for (int t = pair; t < total; t += npairs, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            const Tile tl = tile_of(t);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, kDevTimeout);
                }
                break;
            }
            tc_fence_after();
            const int row0 = tl.a_row + static_cast<int>(rank) * kHalf + q * 32;
            const int n0 = tl.n0;
            const bool whole = !GROUPED || row0 + 32 <= tl.row_end;     // warp-uniform
            const int64_t row = static_cast<int64_t>(row0) + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
            if (row0 < tl.row_end) {
#pragma unroll 1
                for (int bx = 0; bx < kOutTile / kOutCols && n0 + bx * kOutCols < p.N; ++bx) {
                    uint32_t r[32], w[32];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        // debug build: the columns read lie inside this CTA's two accumulators
                        (void)BI_IN_BOUNDS(acc * kBN + bx * kOutCols + hf * 32 + 32 + (SILU ? kOutTile : 0) <= kTmemCols,
                                           p.status);
                        tmem_ld_32x32b_x32(taddr + bx * kOutCols + hf * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[16 * hf + i] = pack_bf16x2(r[2 * i], r[2 * i + 1]);
                        if constexpr (SILU) {   // the matching up columns sit kOutTile columns further
                            tmem_ld_32x32b_x32(taddr + kOutTile + bx * kOutCols + hf * 32, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[16 * hf + i] = silu_mul_bf16x2(w[16 * hf + i], pack_bf16x2(r[2 * i], r[2 * i + 1]));
                        }
                    }
                    if (whole) {
                        uint8_t *buf = boxes + (bx % kBoxes) * kOutBytes;
                        if (lane == 0) {      // the box last stored from this buffer has left it
                            if constexpr (kBoxes == 2) bulk_wait_group_read1(); else bulk_wait_group_read0();
                        }
                        __syncwarp();
                        const uint32_t sb = smem_u32(buf) + lane * 128;
#pragma unroll
                        for (int c = 0; c < kOutCols / 8; ++c)
                            st_shared_v4(sb + ((c ^ (lane & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                                         w[4 * c + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmY, buf, n0 + bx * kOutCols, row0);
                            bulk_commit_group();
                        }
                    } else if (row < tl.row_end && BI_IN_BOUNDS(row < p.M, p.status)) {
                        uint8_t *yrow = p.Yg + (row * p.N + n0 + bx * kOutCols) * 2;
#pragma unroll
                        for (int c = 0; c < kOutCols / 8; ++c)
                            if (n0 + bx * kOutCols + c * 8 < p.N)
                                st_global_v4(yrow + c * 16, w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    grid_dep_launch();                   // the next kernel may start launching on SMs as they free up
    tc_fence_before();
    cluster_sync();                      // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

void plan_gemm_bf16_one_segment(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    pl->op = BI_OP_GEMM_BF16;
    pl->block_m = kBM; pl->block_n = kBN; pl->block_k = kBK;
    pl->mma_m = kBM; pl->mma_n = kBN; pl->mma_k = kMmaK;
    pl->k_steps = static_cast<int32_t>((K + kBK - 1) / kBK);
    pl->split_k = 1;
    pl->stages = kStages;
    pl->threads = kThreads;
    pl->smem_bytes = smem_bytes<kDense>();
    pl->tiles_m = (M + kBM - 1) / kBM;
    pl->tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = pl->tiles_m * pl->tiles_n;
    const int64_t pairs = sms / 2;
    pl->grid = static_cast<int32_t>(2 * (tiles < pairs ? tiles : pairs));
    pl->reduce_tree = 0;
}

void plan_grouped_gemm_bf16(int64_t rows, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    pl->op = BI_OP_GROUPED_GEMM_BF16;
    pl->block_m = kBM; pl->block_n = kBN; pl->block_k = kBK;
    pl->mma_m = kBM; pl->mma_n = kBN; pl->mma_k = kMmaK;
    pl->k_steps = static_cast<int32_t>((K + kBK - 1) / kBK);
    pl->split_k = 1;
    pl->stages = kStages;
    pl->threads = kThreads;
    pl->smem_bytes = smem_bytes<kGrouped>();
    pl->tiles_m = (rows + kBM - 1) / kBM;   // without the per-expert partial tiles
    pl->tiles_n = (N + kBN - 1) / kBN;
    pl->grid = sms / 2 * 2;                 // the tile count is only known on the device
    pl->reduce_tree = 0;
}

template <int MODE>
bi_status launch_pair(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ty, const Params &p, int grid,
                      cudaStream_t s) {
    static unsigned long long configured = 0;
    auto kern = gemm_bf16_pair_kernel<MODE>;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), smem_bytes<MODE>(), &configured) != BI_OK)
        return BI_ERR_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem_bytes<MODE>(), s, ta, tb, ty, p);
}

bi_status launch_gemm_bf16_one_segment(const void *X, int64_t ldx, const void *W, int64_t ldw, void *Y, int64_t ldy,
                                       int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    // With fewer than 128 rows, each CTA copies only the A rows that can hold
    // data (rounded up to 16); the MMA still multiplies 128 rows, and the
    // accumulator rows past M -- computed from whatever the rest of the tile
    // holds -- are never stored. Rows never interact, so this changes no bit
    // of any stored row; it only spares the copy engine the zero rows.
    const int a_rows = M >= kHalf ? kHalf : static_cast<int>((M + 15) / 16 * 16);
    CUtensorMap ta, tb, ty;
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, ldx * 2, kBK, a_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, K, N, ldw * 2, kBK, kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, N, M, ldy * 2, kOutCols, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    bi_plan_t pl;
    plan_gemm_bf16_one_segment(M, N, K, info->sm_count, &pl);
    Params p{};
    p.a_bytes = a_rows * kBK * 2;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.status = device_status_word();
    return launch_pair<kDense>(ta, tb, ty, p, pl.grid, s);
}

// Grouped launch. silu == false: Y [rows][N] = X W[e]^T with W [E][N][K].
// silu == true: W [E][2N][K] holds each expert's gate rows then its up rows,
// and Y [rows][N] = bf16(silu(gate) * up) with gate and up rounded to bf16.
bi_status launch_grouped(const void *X, const void *W, void *Y, const int32_t *offsets, int32_t E, int64_t rows,
                         int64_t N, int64_t K, bool silu, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    if (E > kMaxExperts) return BI_ERR_INVALID_ARG;
    CUtensorMap ta, tb, ty;
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, rows, K * 2, kBK, kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, K, static_cast<uint64_t>(E) * N * (silu ? 2 : 1), K * 2,
                      kBK, kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, N, rows, N * 2, kOutCols, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    Params p{};
    p.a_bytes = kABytes;
    p.M = static_cast<int32_t>(rows);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.offsets = offsets;
    p.E = E;
    p.Yg = static_cast<uint8_t *>(Y);
    p.status = device_status_word();
    // Upper bound on tiles: every expert adds at most one partial 256-row tile.
    const int64_t out_tile = silu ? kBN / 2 : kBN;
    const int64_t tiles_n = (N + out_tile - 1) / out_tile;
    const int64_t max_tiles = ((rows + kBM - 1) / kBM + E) * tiles_n;
    const int64_t pairs = info->sm_count / 2;
    const int grid = static_cast<int>(2 * (max_tiles < pairs ? max_tiles : pairs));
    return silu ? launch_pair<kGroupedSilu>(ta, tb, ty, p, grid, s) : launch_pair<kGrouped>(ta, tb, ty, p, grid, s);
}

bi_status launch_grouped_gemm_bf16(const void *X, const void *W, void *Y, const int32_t *offsets, int32_t E,
                                   int64_t rows, int64_t N, int64_t K, cudaStream_t s) {
    return launch_grouped(X, W, Y, offsets, E, rows, N, K, false, s);
}

bi_status launch_grouped_gemm_silu_bf16(const void *X, const void *W, void *act, const int32_t *offsets, int32_t E,
                                        int64_t rows, int64_t I, int64_t K, cudaStream_t s) {
    return launch_grouped(X, W, act, offsets, E, rows, I, K, true, s);
}

}  // namespace bi
