// gemm_nvfp4_pair.cu -- batch-invariant block-scaled NVFP4 linear layer on CTA pairs.
//
// Y[i][j] = bf16( alpha * sum_k (a[i][k] sa[i][k/16]) (b[j][k] sb[j][k/16]) ), the
// NVFP4 linear layer of vLLM PR #39912 ("NVFP4 CUTLASS batch invariant mode").
//
// 256 x 256 output tiles on clusters of two CTAs (one per SM), K stages of 256
// e2m1 values (128 bytes per row), 5 stages of 38 KB per CTA:
//   - warp 0 of each CTA TMA-loads its own 128 rows of A, its half (128 rows)
//     of B, the scale atoms of its own A rows (4 x 512 bytes) and the scale
//     atoms of all 256 B rows (8 x 512 bytes; tiny, so both CTAs load them);
//     every copy completes on the leader CTA's "full" barrier (cta_group::2);
//   - one thread of the leader copies each stage's scale atoms from each CTA's
//     shared memory into that CTA's tensor memory (tcgen05.cp.cta_group::2,
//     32 lanes x 128 bits replicated to the four lane quarters: lane l,
//     column c holds row 32c + l), then issues four
//     tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X
//     (256 x 256 x 64, fp32 accumulate): each SM's tensor core multiplies its
//     128 A rows by both B halves;
//   - both CTAs' epilogue warps read their own accumulator rows, scale by
//     alpha, round to bf16, hand the accumulator back to the leader, then store.
// Per FLOP this issues half the scale-factor copies and loads half the operand
// bytes of the single-CTA 128 x 256 tile.
//
// TMEM per CTA: one 256-column accumulator + a 5 x 48-column scale ring.
// Invariance: tile shape, MMA shape and K order (ascending 64-wide steps from
// zero) are the same for every M; rows never interact.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kBM = 256;                 // pair tile rows (128 per CTA)
constexpr int kHalf = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;            // K bytes per stage (256 e2m1 values)
constexpr int kBK = 2 * kBKBytes;
constexpr int kMmaK = 64;
constexpr int kMmasPerStage = kBK / kMmaK;
constexpr int kStages = 5;
constexpr int kThreads = 192;
constexpr int kGroupM = 8;
constexpr int kAtom = 512;

constexpr int kABytes = kHalf * kBKBytes;                   // 16 KB
constexpr int kBBytes = kHalf * kBKBytes;                   // 16 KB (this CTA's half)
constexpr int kSfaBytes = kMmasPerStage * kAtom;            // 2 KB
constexpr int kSfbBytes = 2 * kMmasPerStage * kAtom;        // 4 KB (both B row blocks)
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
constexpr int kBarBytes = 256;
constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;

constexpr int kTmemCols = 512;
constexpr int kAccCol = 0;
constexpr int kSfCol = 256;
constexpr int kSfColsPerMma = 4 + 8;
constexpr int kSfColsPerStage = kMmasPerStage * kSfColsPerMma;
static_assert(kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

struct Params {
    uint8_t *Y;
    float alpha;
    int32_t M, N, K;
    int32_t atoms_per_rowblock;   // K / 64
    unsigned *status;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemm_nvfp4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                       const Params p) {
    constexpr uint32_t kIdesc = idesc_nvf4(kBM, kBN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;
    uint64_t *tempty = tfull + 1;
    uint64_t *drain = tempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    auto stage_a = [&](int s) { return smem + s * kStageBytes; };
    auto stage_b = [&](int s) { return smem + s * kStageBytes + kABytes; };
    auto stage_sfa = [&](int s) { return smem + s * kStageBytes + kABytes + kBBytes; };
    auto stage_sfb = [&](int s) { return smem + s * kStageBytes + kABytes + kBBytes + kSfaBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
    const int num_m = (p.M + kBM - 1) / kBM;
    const int num_n = (p.N + kBN - 1) / kBN;
    const int total = num_m * num_n;
    const int k_stages = (p.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 8);            // 4 epilogue warps in each CTA
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSFA);
        tma_prefetch_desc(&tmSFB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto tile_of = [&](int t, int &mb, int &nb) {
        const int per_group = kGroupM * num_n;
        const int g = t / per_group;
        const int first = g * kGroupM;
        const int gm = min(kGroupM, num_m - first);
        const int local = t - g * per_group;
        mb = first + local % gm;
        nb = local / gm;
    };
    auto mmas_in = [&](int ks) { return min(kMmasPerStage, (p.K - ks * kBK) / kMmaK); };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                int mb, nb;
                tile_of(t, mb, nb);
                const int a_row = mb * kBM + static_cast<int>(rank) * kHalf;
                const int b_row = nb * kBN + static_cast<int>(rank) * kHalf;
                const int rb_a = mb * 2 + static_cast<int>(rank);       // this CTA's 128-row scale block
                const int rb_b = nb * 2;                                 // the tile's two B scale blocks
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
                    const uint32_t bar = full_leader + stage * 8;
                    const int atom = ks * kMmasPerStage;
                    tma_load_2d_pair_bar(stage_a(stage), &tmA, bar, ks * kBKBytes, a_row);
                    tma_load_2d_pair_bar(stage_b(stage), &tmB, bar, ks * kBKBytes, b_row);
                    tma_load_3d_pair_bar(stage_sfa(stage), &tmSFA, bar, 0, 0, rb_a * p.atoms_per_rowblock + atom);
                    tma_load_3d_pair_bar(stage_sfb(stage), &tmSFB, bar, 0, 0, rb_b * p.atoms_per_rowblock + atom);
                    tma_load_3d_pair_bar(stage_sfb(stage) + kMmasPerStage * kAtom, &tmSFB, bar, 0, 0,
                                         (rb_b + 1) * p.atoms_per_rowblock + atom);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            for (int i = 0; i < kStages && ok; ++i) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) ok = false;
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                if (rank == 0)   // the leader's full barriers count both CTAs' bytes
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
            const uint32_t d = tmem_base + kAccCol;
            for (int t = pair; t < total && ok; t += npairs, ++it) {
                if (!mbar_wait(tempty, (it & 1) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const int nk = mmas_in(ks);
                    const uint32_t sf = tmem_base + kSfCol + stage * kSfColsPerStage;
                    const uint32_t sa = smem_u32(stage_sfa(stage)), sb = smem_u32(stage_sfb(stage));
                    for (int j = 0; j < nk; ++j) {
                        tmem_cp_32x128b_x4_pair(sf + j * kSfColsPerMma, sdesc_plain_128(sa + j * kAtom));
                        tmem_cp_32x128b_x4_pair(sf + j * kSfColsPerMma + 4, sdesc_plain_128(sb + j * kAtom));
                        tmem_cp_32x128b_x4_pair(sf + j * kSfColsPerMma + 8,
                                                sdesc_plain_128(sb + (kMmasPerStage + j) * kAtom));
                    }
                    const uint32_t a0 = smem_u32(stage_a(stage)), b0 = smem_u32(stage_b(stage));
                    for (int j = 0; j < nk; ++j)
                        mma_nvf4_pair(d, sdesc_k_sw128(a0 + j * (kMmaK / 2)), sdesc_k_sw128(b0 + j * (kMmaK / 2)),
                                      kIdesc, sf + j * kSfColsPerMma, sf + j * kSfColsPerMma + 4, (ks | j) != 0);
                    tc_commit_pair(&empty[stage], 0x3);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(tfull, 0x3);
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
        const int q = warp & 3;
        const int r_in_tile = static_cast<int>(rank) * kHalf + q * 32 + lane;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        int it = 0;
        for (int t = pair; t < total; t += npairs, ++it) {
            int mb, nb;
            tile_of(t, mb, nb);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(tfull, it & 1, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, kDevTimeout);
                }
                break;
            }
            tc_fence_after();
            uint32_t packed[kBN / 2];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[c * 16 + i] = pack_bf16x2(__float_as_uint(__uint_as_float(r[2 * i]) * p.alpha),
                                                     __float_as_uint(__uint_as_float(r[2 * i + 1]) * p.alpha));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader);   // accumulator may be overwritten now
            const int64_t row = static_cast<int64_t>(mb) * kBM + r_in_tile;
            if (row < p.M) {
                const int n0 = nb * kBN;
                uint8_t *yrow = p.Y + (row * p.N + n0) * 2;
#pragma unroll
                for (int g = 0; g < kBN / 8; ++g)
                    if (n0 + g * 8 < p.N)
                        st_global_v4(yrow + g * 16, packed[4 * g], packed[4 * g + 1], packed[4 * g + 2],
                                     packed[4 * g + 3]);
            }
        }
    }

    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

void plan_gemm_nvfp4(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    pl->op = BI_OP_GEMM_NVFP4;
    pl->block_m = kBM; pl->block_n = kBN; pl->block_k = kBK;
    pl->mma_m = kBM; pl->mma_n = kBN; pl->mma_k = kMmaK;
    pl->k_steps = static_cast<int32_t>((K + kMmaK - 1) / kMmaK);
    pl->split_k = 1;
    pl->stages = kStages;
    pl->threads = kThreads;
    pl->smem_bytes = kSmem;
    pl->tiles_m = (M + kBM - 1) / kBM;
    pl->tiles_n = (N + kBN - 1) / kBN;
    const int64_t tiles = pl->tiles_m * pl->tiles_n, pairs = sms / 2;
    pl->grid = static_cast<int32_t>(2 * (tiles < pairs ? tiles : pairs));
    pl->reduce_tree = 0;
}

bi_status launch_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B, const uint8_t *B_sf,
                            float alpha, void *Y, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    CUtensorMap ta, tb, tsa, tsb;
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K / 2, M, K / 2, kBKBytes, kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K / 2, N, K / 2, kBKBytes, kHalf, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    // Scale atoms viewed as [atoms][2][256] bytes: one box = 4 atoms = one K stage of one 128-row block.
    const uint64_t per_rb = static_cast<uint64_t>(K / 64);
    const uint64_t sfa_dims[3] = {256, 2, static_cast<uint64_t>((M + 127) / 128) * per_rb};
    const uint64_t sfb_dims[3] = {256, 2, static_cast<uint64_t>((N + 127) / 128) * per_rb};
    const uint64_t sf_strides[2] = {256, 512};
    const uint32_t sf_box[3] = {256, 2, kMmasPerStage};
    st = make_tmap_3d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, A_sf, sfa_dims, sf_strides, sf_box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != BI_OK) return st;
    st = make_tmap_3d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B_sf, sfb_dims, sf_strides, sf_box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != BI_OK) return st;
    bi_plan_t pl;
    plan_gemm_nvfp4(M, N, K, info->sm_count, &pl);
    Params p{};
    p.Y = static_cast<uint8_t *>(Y);
    p.alpha = alpha;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.atoms_per_rowblock = static_cast<int32_t>(K / 64);
    p.status = device_status_word();
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(gemm_nvfp4_pair_kernel), kSmem, &configured) != BI_OK)
        return BI_ERR_CUDA;
    gemm_nvfp4_pair_kernel<<<pl.grid, kThreads, kSmem, s>>>(ta, tb, tsa, tsb, p);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace bi
