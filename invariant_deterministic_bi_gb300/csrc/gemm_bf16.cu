// gemm_bf16.cu -- batch-invariant MoE-grouped bf16 linear layers on tcgen05 (single-CTA tiles).
//
// (Dense Y = X W^T uses the CTA-pair kernel in gemm_bf16_pair.cu; expert groups
// are often a few hundred rows, where 128-row tiles waste less.)
// One persistent, warp-specialised kernel per (BN, stages) configuration:
//   warp 0      TMA producer: A tile [128 x 64] and B tile [BN x 64] per K step
//               into a STAGES-deep shared-memory ring (128-byte swizzle);
//   warp 1      MMA issuer: one thread issues 4 x tcgen05.mma (128 x BN x 16,
//               bf16 in, fp32 accumulate) per K step into a TMEM accumulator;
//               two accumulators (2 x BN columns) let the epilogue of tile i
//               overlap the main loop of tile i+1;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns, fp32 -> bf16 RNE,
//               16-byte stores of the rows that exist.
//
// Batch invariance (vLLM PR #39912, "NVFP4 CUTLASS batch invariant mode":
// a fixed persistent tile schedule, no M-dependent configuration): the tile
// shape, MMA shape and K loop depend only on (N, K). Every output element is
// accumulated by exactly one CTA in ascending K order (K steps of 64, four
// 16-wide MMA steps each), starting from zero. Rows of the 128-row tile never
// interact, so row i of Y is the same bits whatever M is, where the row sits
// in the batch and whatever the padding rows (or, for the grouped case, the
// rows of the next expert) contain. Only which CTA computes which tile, and
// when, depends on M; that changes nothing in any element.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kBM = 128;      // tile rows = MMA M (cta_group::1)
constexpr int kBK = 64;       // K step: 64 bf16 = one 128-byte swizzle row
constexpr int kMmaK = 16;     // K per tcgen05.mma (kind::f16)
constexpr int kThreads = 192; // 6 warps
constexpr int kGroupM = 16;   // tile raster: 16 M-tiles per band for L2 reuse
constexpr int kMaxExperts = 1024;

template <int BN, int STAGES>
struct Cfg {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kBarBytes = 256;
    static constexpr int kSchedBytes = 2 * (kMaxExperts + 1) * 4 + 16;
    static constexpr int kSmem = 1024 + STAGES * kStageBytes + kBarBytes + kSchedBytes;
    static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "MMA N");
};

struct Params {
    uint8_t *Y;
    int64_t ldy;               // elements
    int32_t M;                 // dense: rows of X / Y
    int32_t N, K;
    const int32_t *offsets;    // grouped: device offsets [E+1]
    int32_t E;
    int32_t rows;              // grouped: offsets[E]
    unsigned *status;
};

struct Tile {
    int32_t a_row;     // first row of the A tile (TMA coordinate)
    int32_t row_end;   // rows >= row_end of this tile are not stored
    int32_t n0;        // first output column
    int32_t b_row;     // first row of the B tile (TMA coordinate)
};

__device__ __forceinline__ Tile dense_tile(int t, int num_m, int num_n, const Params &p, int bn) {
    const int per_group = kGroupM * num_n;
    const int g = t / per_group;
    const int first = g * kGroupM;
    const int gm = min(kGroupM, num_m - first);
    const int local = t - g * per_group;
    const int mb = first + local % gm, nb = local / gm;
    return Tile{mb * kBM, p.M, nb * bn, nb * bn};
}

// Grouped raster: experts in order; inside an expert, M-tiles fastest so the
// CTAs working at the same time share the expert's weight panel in L2.
__device__ __forceinline__ Tile grouped_tile(int t, int num_n, const int *off_s, const int *pre_s,
                                             const Params &p, int bn) {
    const int x = t / num_n;
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre_s[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int mt = pre_s[e + 1] - pre_s[e];
    const int local = t - pre_s[e] * num_n;
    const int mb = local % mt, nb = local / mt;
    return Tile{off_s[e] + mb * kBM, off_s[e + 1], nb * bn, e * p.N + nb * bn};
}

template <int BN, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
    using C = Cfg<BN, STAGES>;
    constexpr uint32_t kIdesc = idesc_bf16(kBM, BN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * C::kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * C::kStageBytes);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *total_s = reinterpret_cast<int *>(tmem_slot + 2);
    int *off_s = reinterpret_cast<int *>(smem + STAGES * C::kStageBytes + C::kBarBytes);
    int *pre_s = off_s + (kMaxExperts + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_n = (p.N + BN - 1) / BN;
    const int k_steps = (p.K + kBK - 1) / kBK;
    const int num_m = GROUPED ? 0 : (p.M + kBM - 1) / kBM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
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
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if constexpr (GROUPED) {
        for (int i = threadIdx.x; i <= p.E; i += kThreads) off_s[i] = p.offsets[i];
        __syncthreads();
        if (threadIdx.x == 0) {
            bool ok = off_s[0] == 0 && off_s[p.E] == p.rows;
            int acc = 0;
            pre_s[0] = 0;
            for (int e = 0; e < p.E; ++e) {
                const long long c = static_cast<long long>(off_s[e + 1]) - off_s[e];
                if (c < 0) ok = false;
                acc += ok ? static_cast<int>((c + kBM - 1) / kBM) : 0;
                pre_s[e + 1] = acc;
            }
            *total_s = ok ? acc * num_n : 0;
            if (!ok && blockIdx.x == 0) atomicOr(p.status, kDevBadOffsets);
        }
    } else {
        if (threadIdx.x == 0) *total_s = num_m * num_n;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = *total_s;

    auto tile_of = [&](int t) -> Tile {
        if constexpr (GROUPED) return grouped_tile(t, num_n, off_s, pre_s, p, BN);
        else return dense_tile(t, num_m, num_n, p, BN);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                for (int kb = 0; kb < k_steps; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                    tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kb * kBK, tl.a_row);
                    tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kb * kBK, tl.b_row);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Tail: wait until every stage has been released by the MMAs.
            for (int i = 0; i < STAGES && ok; ++i) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) ok = false;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                for (int s = 0; s < STAGES; ++s)   // let copies in flight land
                    if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_phase >> s) & 1u, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < k_steps; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * C::kABytes);
                    const uint32_t b0 = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / kMmaK; ++k)
                        mma_bf16(d, sdesc_k_sw128(a0 + k * kMmaK * 2), sdesc_k_sw128(b0 + k * kMmaK * 2), kIdesc,
                                 (kb | k) != 0);
                    tc_commit(&empty[stage]);   // frees the stage when these MMAs finish
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);          // accumulator ready for the epilogue
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                tc_commit(drain);                // wait for the MMAs already issued
                mbar_wait(drain, 0, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        const int r_in_tile = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
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
            const int64_t row = static_cast<int64_t>(tl.a_row) + r_in_tile;
            const bool valid = row < tl.row_end;
            uint8_t *yrow = p.Y + (row * p.ldy + tl.n0) * 2;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (tl.n0 + c * 32 + g * 8 < p.N)
                            st_global_v4(yrow + (c * 32 + g * 8) * 2, pack_bf16x2(r[8 * g + 0], r[8 * g + 1]),
                                         pack_bf16x2(r[8 * g + 2], r[8 * g + 3]),
                                         pack_bf16x2(r[8 * g + 4], r[8 * g + 5]),
                                         pack_bf16x2(r[8 * g + 6], r[8 * g + 7]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// The one configuration used for every (N, K): BN = 256, 4 stages.
constexpr int kBN = 256;
constexpr int kStages = 4;

template <bool GROUPED>
bi_status launch(const CUtensorMap &ta, const CUtensorMap &tb, const Params &p, int grid, cudaStream_t s) {
    using C = Cfg<kBN, kStages>;
    auto kern = gemm_bf16_kernel<kBN, kStages, GROUPED>;
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::kSmem, &configured) != BI_OK) return BI_ERR_CUDA;
    kern<<<grid, kThreads, C::kSmem, s>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace

void plan_grouped_gemm_bf16(int64_t rows, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    using C = Cfg<kBN, kStages>;
    pl->op = BI_OP_GROUPED_GEMM_BF16;
    pl->block_m = kBM; pl->block_n = kBN; pl->block_k = kBK;
    pl->mma_m = kBM; pl->mma_n = kBN; pl->mma_k = kMmaK;
    pl->k_steps = static_cast<int32_t>((K + kBK - 1) / kBK);
    pl->split_k = 1;
    pl->stages = kStages;
    pl->threads = kThreads;
    pl->smem_bytes = C::kSmem;
    pl->tiles_m = (rows + kBM - 1) / kBM;   // without the per-expert partial tiles
    pl->tiles_n = (N + kBN - 1) / kBN;
    pl->grid = sms;                         // the tile count is only known on the device
    pl->reduce_tree = 0;
}

bi_status launch_grouped_gemm_bf16(const void *X, const void *W, void *Y, const int32_t *offsets, int32_t E,
                                   int64_t rows, int64_t N, int64_t K, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    CUtensorMap ta, tb;
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, rows, K * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, K, static_cast<uint64_t>(E) * N, K * 2, kBK, kBN,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    Params p{};
    p.Y = static_cast<uint8_t *>(Y);
    p.ldy = N;
    p.M = 0;
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.offsets = offsets;
    p.E = E;
    p.rows = static_cast<int32_t>(rows);
    p.status = device_status_word();
    // Upper bound on tiles: every expert adds at most one partial M-tile.
    const int64_t tiles_n = (N + kBN - 1) / kBN;
    const int64_t max_tiles = ((rows + kBM - 1) / kBM + E) * tiles_n;
    const int grid = static_cast<int>(max_tiles < info->sm_count ? max_tiles : info->sm_count);
    return launch<true>(ta, tb, p, grid, s);
}

}  // namespace bi
