// gemm_nvfp4.cu -- batch-invariant block-scaled NVFP4 linear layer on tcgen05.
//
// Y[i][j] = bf16( alpha * sum_k (a[i][k] sa[i][k/16]) (b[j][k] sb[j][k/16]) ), the
// NVFP4 linear layer of vLLM PR #39912 ("NVFP4 CUTLASS batch invariant mode"):
// e2m1 values two per byte, one e4m3 scale per 16 K elements, alpha = 1/(gsA gsB).
//
// Persistent, warp-specialised, one configuration for every M:
//   warp 0      producer: per K stage of 256 elements (128 bytes per row, one
//               128-byte swizzle row) TMA-loads the A tile [128 x 128 B] and
//               B tile [256 x 128 B], and bulk-copies the stage's scale atoms
//               (512 bytes = 128 rows x 4 scales each) from the interleaved
//               scale buffers;
//   warp 1      MMA issuer: copies the stage's scale atoms from shared to
//               tensor memory (tcgen05.cp 32x128b, replicated to the four lane
//               quarters) into that stage's TMEM scale slot, then issues four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (128 x 256
//               x 64, fp32 accumulate) in ascending K;
//   warps 2..5  epilogue: read the accumulator, scale by alpha, round to bf16,
//               release the accumulator, then store.
// TMEM: one 256-column accumulator + a 4 x 48-column scale ring (A: 4 columns,
// B: 8 columns per MMA). The accumulator is handed back to the MMA thread as
// soon as the epilogue holds it in registers, so the next tile's main loop
// overlaps the stores.
//
// Invariance: tile shape, MMA shape and K order depend on nothing; each output
// element is accumulated by one CTA from zero in ascending K; rows never mix.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;            // K bytes per stage (256 e2m1 values)
constexpr int kBK = 2 * kBKBytes;        // K elements per stage
constexpr int kMmaK = 64;                // K per MMA
constexpr int kMmasPerStage = kBK / kMmaK;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kGroupM = 16;
constexpr int kAtom = 512;               // 128 rows x 4 scales

constexpr int kABytes = kBM * kBKBytes;                     // 16 KB
constexpr int kBBytes = kBN * kBKBytes;                     // 32 KB
constexpr int kSfaBytes = kMmasPerStage * kAtom;            // 2 KB
constexpr int kSfbBytes = 2 * kMmasPerStage * kAtom;        // 4 KB (two 128-row blocks)
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
constexpr int kBarBytes = 256;
constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes;

constexpr int kTmemCols = 512;
constexpr int kAccCol = 0;                                  // 256 columns
constexpr int kSfCol = 256;                                 // scale ring
constexpr int kSfColsPerMma = 4 + 8;
constexpr int kSfColsPerStage = kMmasPerStage * kSfColsPerMma;   // 48
static_assert(kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

struct Params {
    uint8_t *Y;
    const uint8_t *sfa;
    const uint8_t *sfb;
    float alpha;
    int32_t M, N, K;
    int32_t atoms_per_rowblock;   // K / 64
    int32_t sfb_rowblocks;        // ceil(N / 128)
    unsigned *status;
};

__global__ void __launch_bounds__(kThreads, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
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
        mbar_init(tempty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
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
    // MMAs in K stage ks (the last stage may hold fewer than four).
    auto mmas_in = [&](int ks) { return min(kMmasPerStage, (p.K - ks * kBK) / kMmaK); };

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int mb, nb;
                tile_of(t, mb, nb);
                const int rb_b = nb * 2;
                const bool two_b = rb_b + 1 < p.sfb_rowblocks;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    const int nk = mmas_in(ks);
                    const uint32_t sf_bytes = static_cast<uint32_t>(nk * kAtom);
                    mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes + sf_bytes * (two_b ? 3u : 2u));
                    tma_load_2d(stage_a(stage), &tmA, &full[stage], ks * kBKBytes, mb * kBM);
                    tma_load_2d(stage_b(stage), &tmB, &full[stage], ks * kBKBytes, nb * kBN);
                    const int64_t atom0 = static_cast<int64_t>(ks) * kMmasPerStage;
                    bulk_load(stage_sfa(stage), p.sfa + (static_cast<int64_t>(mb) * p.atoms_per_rowblock + atom0) * kAtom,
                              sf_bytes, &full[stage]);
                    bulk_load(stage_sfb(stage), p.sfb + (static_cast<int64_t>(rb_b) * p.atoms_per_rowblock + atom0) * kAtom,
                              sf_bytes, &full[stage]);
                    if (two_b)
                        bulk_load(stage_sfb(stage) + kMmasPerStage * kAtom,
                                  p.sfb + (static_cast<int64_t>(rb_b + 1) * p.atoms_per_rowblock + atom0) * kAtom,
                                  sf_bytes, &full[stage]);
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
                for (int s = 0; s < kStages; ++s)
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
            const uint32_t d = tmem_base + kAccCol;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                if (!mbar_wait(tempty, (it & 1) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const int nk = mmas_in(ks);
                    const uint32_t sf = tmem_base + kSfCol + stage * kSfColsPerStage;
                    const uint32_t sa = smem_u32(stage_sfa(stage)), sb = smem_u32(stage_sfb(stage));
                    for (int j = 0; j < nk; ++j) {
                        tmem_cp_32x128b_x4(sf + j * kSfColsPerMma, sdesc_plain_128(sa + j * kAtom));
                        tmem_cp_32x128b_x4(sf + j * kSfColsPerMma + 4, sdesc_plain_128(sb + j * kAtom));
                        tmem_cp_32x128b_x4(sf + j * kSfColsPerMma + 8,
                                           sdesc_plain_128(sb + (kMmasPerStage + j) * kAtom));
                    }
                    const uint32_t a0 = smem_u32(stage_a(stage)), b0 = smem_u32(stage_b(stage));
                    for (int j = 0; j < nk; ++j)
                        mma_nvf4(d, sdesc_k_sw128(a0 + j * (kMmaK / 2)), sdesc_k_sw128(b0 + j * (kMmaK / 2)), kIdesc,
                                 sf + j * kSfColsPerMma, sf + j * kSfColsPerMma + 4, (ks | j) != 0);
                    tc_commit(&empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(tfull);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kDevTimeout);
                tc_commit(drain);
                mbar_wait(drain, 0, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
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
            if (lane == 0) mbar_arrive(tempty);     // the accumulator may be overwritten now
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
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
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
    const int64_t tiles = pl->tiles_m * pl->tiles_n;
    pl->grid = static_cast<int32_t>(tiles < sms ? tiles : sms);
    pl->reduce_tree = 0;
}

bi_status launch_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B, const uint8_t *B_sf,
                            float alpha, void *Y, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    CUtensorMap ta, tb;
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K / 2, M, K / 2, kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    st = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K / 2, N, K / 2, kBKBytes, kBN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    bi_plan_t pl;
    plan_gemm_nvfp4(M, N, K, info->sm_count, &pl);
    Params p{};
    p.Y = static_cast<uint8_t *>(Y);
    p.sfa = A_sf;
    p.sfb = B_sf;
    p.alpha = alpha;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.atoms_per_rowblock = static_cast<int32_t>(K / kMmaK);
    p.sfb_rowblocks = static_cast<int32_t>((N + 127) / 128);
    p.status = device_status_word();
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(gemm_nvfp4_kernel), kSmem, &configured) != BI_OK)
        return BI_ERR_CUDA;
    gemm_nvfp4_kernel<<<pl.grid, kThreads, kSmem, s>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

}  // namespace bi
