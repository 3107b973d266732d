// gemm_nvfp4.cu -- batch-invariant block-scaled NVFP4 linear layer.
//
// Y[i][j] = bf16( alpha * sum_k (a[i][k] sa[i][k/16]) (b[j][k] sb[j][k/16]) ), the
// NVFP4 linear layer of vLLM PR #39912 ("NVFP4 CUTLASS batch invariant mode").
//
// Output tiles are 256 x 256, each computed by a CTA pair (a cluster of two
// CTAs, cta_group::2, one CTA per SM, 128 accumulator rows each). Every CTA
// loads its own operands with plain TMA copies into its own shared memory:
// the 128 A rows of its lane half and its 128-row half of the B tile. K
// advances in stages of 256 e2m1 values (128 bytes per row), 5 stages of
// 38 KB per CTA. Warp roles:
//   - warp 0 (both CTAs): per stage, its 128 A rows, its 128 B rows and the
//     stage's scale atoms (its 4 A atoms, all 8 B atoms of the pair's tile,
//     512 bytes each), all counted on its own "full" barrier;
//   - warps 2-5 (both CTAs): one per tensor-memory lane quarter; once "full"
//     completes they move the scale atoms from shared memory into the
//     stage's scale slot in tensor memory with tcgen05.st (each quarter holds
//     the same 48 columns: lane l, column c = row 32c + l of an atom), wait
//     for the stores and report to the pair leader's "ready" barrier -- so
//     "ready" also means both CTAs' operands have landed;
//   - warp 1 (pair leader): one thread issues four
//     tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X
//     (256 x 256 x 64, fp32 accumulate) per stage, then commits the stage to
//     both CTAs' "empty" barriers;
//   - warps 6-13 (both CTAs): two warps per lane quarter, 128 columns each:
//     read the accumulator, scale by alpha, round to bf16, hand the
//     accumulator back, then write 32 x 64 boxes through a swizzled staging
//     buffer with TMA stores (rows past M, columns past N are clipped).
// Writing the scales with tcgen05.st keeps them off the tensor pipe: the
// equivalent twelve tcgen05.cp 32x128b copies per stage cost more tensor-pipe
// time than the stage's four MMAs.
//
// TMEM per CTA: one 256-column accumulator + a 5 x 48-column scale ring.
// Invariance: tile shape, MMA shape and K order (ascending 64-wide steps from
// zero) are the same for every M; rows never interact; which pair computes
// which tile does not change any result.
#include <cuda_bf16.h>

#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kClusterCtas = 2;          // one CTA pair
constexpr int kBM = 256;                 // pair tile rows (128 per CTA)
constexpr int kHalf = 128;               // A rows and B rows each CTA loads per stage
constexpr int kBN = 256;
constexpr int kBKBytes = 128;            // K bytes per stage (256 e2m1 values)
constexpr int kBK = 2 * kBKBytes;
constexpr int kMmaK = 64;
constexpr int kMmasPerStage = kBK / kMmaK;
constexpr int kStages = 5;
constexpr int kSfWarps = 4;              // scale writers, one per TMEM lane quarter
constexpr int kEpiWarps = 8;             // two per lane quarter
constexpr int kThreads = 32 * (2 + kSfWarps + kEpiWarps);
constexpr int kGroupM = 8;
constexpr int kAtom = 512;

constexpr int kABytes = kHalf * kBKBytes;                   // 16 KB (this CTA's 128 A rows)
constexpr int kBBytes = kHalf * kBKBytes;                   // 16 KB (this CTA's half of the pair's B)
constexpr int kSfaBytes = kMmasPerStage * kAtom;            // 2 KB
constexpr int kSfbBytes = 2 * kMmasPerStage * kAtom;        // 4 KB (both B row blocks)
constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
constexpr int kOutCols = 64;                                // bf16 columns per output box (128 bytes)
constexpr int kOutBytes = 32 * kOutCols * 2;                // one epilogue warp's staging box: 32 rows
constexpr int kBarBytes = 256;
constexpr int kSmem = 1024 + kStages * kStageBytes + kEpiWarps * kOutBytes + kBarBytes;

constexpr int kTmemCols = 512;
constexpr int kAccCol = 0;
constexpr int kSfCol = 256;
constexpr int kSfColsPerMma = 4 + 8;     // SFA (128 rows) + SFB (256 rows) per 64-wide K step
constexpr int kSfColsPerStage = kMmasPerStage * kSfColsPerMma;
static_assert(kSfCol + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

struct Params {
    float alpha;
    int32_t M, N, K;
    int32_t atoms_per_rowblock;   // K / 64
    int32_t stage_tx;             // bytes landing in a CTA per stage (fewer A rows when M < 128)
    unsigned *status;
};

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kThreads, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                  const __grid_constant__ CUtensorMap tmY, const Params p) {
    constexpr uint32_t kIdesc = idesc_nvf4(kBM, kBN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *out_stage = smem + kStages * kStageBytes;   // kEpiWarps staging boxes of kOutBytes
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kEpiWarps * kOutBytes);
    uint64_t *empty = full + kStages;        // stage read by the pair's MMAs
    uint64_t *ready = empty + kStages;       // (pair leader) both CTAs' operands and scales in place
    uint64_t *tfull = ready + kStages;
    uint64_t *tempty = tfull + 1;
    uint64_t *drain = tempty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    static_assert((3 * kStages + 3) * 8 + 8 <= kBarBytes, "barrier area");

    auto stage_a = [&](int s) { return smem + s * kStageBytes; };
    auto stage_b = [&](int s) { return smem + s * kStageBytes + kABytes; };
    auto stage_sfa = [&](int s) { return smem + s * kStageBytes + kABytes + kBBytes; };
    auto stage_sfb = [&](int s) { return smem + s * kStageBytes + kABytes + kBBytes + kSfaBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int h = static_cast<int>(rank);               // lane half of the pair's tile (0: leader)
    const int cl = static_cast<int>(blockIdx.x) / kClusterCtas;
    const int ncl = static_cast<int>(gridDim.x) / kClusterCtas;
    const int num_m = (p.M + kBM - 1) / kBM;
    const int num_n = (p.N + kBN - 1) / kBN;
    const int total = num_m * num_n;
    const int k_stages = (p.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&ready[s], 2 * kSfWarps);      // scale writer warps of both CTAs of the pair
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 2 * kEpiWarps);            // epilogue warps of both CTAs of the pair
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
    grid_dep_wait();      // the set-up above overlaps the previous kernel; global memory only from here
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Tile t -> (row tile mb, column tile nb): bands of kGroupM row tiles, row
    // tiles fastest inside a band, so pairs running at the same time share
    // their B panels and A panels in L2.
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
    auto give_up = [&]() {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (every CTA)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = cl; t < total && ok; t += ncl) {
                int mb, nb;
                tile_of(t, mb, nb);
                const int a_row = mb * kBM + h * kHalf;
                const int b_row = nb * kBN + h * kHalf;
                const int rb_a = mb * 2 + h;               // this CTA's 128-row scale block of A
                const int rb_b = nb * 2;                   // the tile's two B scale blocks
                for (int ks = 0; ks < k_stages; ++ks) {
                    // debug build: the copies' coordinates lie inside the operands and scale atoms
                    if (!BI_IN_BOUNDS(ks * kBKBytes < p.K / 2 && a_row < num_m * kBM && b_row < num_n * kBN &&
                                          ks * kMmasPerStage < p.atoms_per_rowblock, p.status)) { ok = false; break; }
                    // the slot is free once the pair's MMAs have read it
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], p.stage_tx);
                    tma_load_2d(stage_a(stage), &tmA, &full[stage], ks * kBKBytes, a_row);
                    tma_load_2d(stage_b(stage), &tmB, &full[stage], ks * kBKBytes, b_row);
                    const int atom = ks * kMmasPerStage;
                    tma_load_3d(stage_sfa(stage), &tmSFA, &full[stage], 0, 0, rb_a * p.atoms_per_rowblock + atom);
                    tma_load_3d(stage_sfb(stage), &tmSFB, &full[stage], 0, 0, rb_b * p.atoms_per_rowblock + atom);
                    tma_load_3d(stage_sfb(stage) + kMmasPerStage * kAtom, &tmSFB, &full[stage], 0, 0,
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
                give_up();
                // let the copies this CTA is waiting for land before it exits
                for (int s = 0; s < kStages; ++s)
                    if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_phase >> s) & 1u, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (pair leader)
        if (lane == 0 && h == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t d = tmem_base + kAccCol;
            for (int t = cl; t < total && ok; t += ncl, ++it) {
                if (!mbar_wait(tempty, (it & 1) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait(&ready[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const int nk = mmas_in(ks);
                    const uint32_t sf = tmem_base + kSfCol + stage * kSfColsPerStage;
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
                give_up();
                tc_commit_pair(drain, 0x1);
                mbar_wait(drain, 0, nullptr);
            }
        }
        __syncwarp();
    } else if (warp < 2 + kSfWarps) {
        // ------------------------------------------------ scale writers (every CTA)
        // Lane l moves 16 bytes per atom: atom bytes l*16 .. l*16+15 are rows
        // l, 32+l, 64+l, 96+l of its 128-row block (4 scales each), i.e. the
        // four 32-bit columns of lane l for that atom.
        const int q = warp & 3;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kSfCol;
        const uint32_t ready_leader = mapa_shared(smem_u32(ready), 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = cl; t < total && ok; t += ncl) {
            for (int ks = 0; ks < k_stages; ++ks) {
                int w = 1;
                if (lane == 0) w = mbar_wait(&full[stage], phase, abort_flag) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    if (lane == 0) give_up();
                    ok = false;
                    break;
                }
                uint32_t r[kSfColsPerStage];
                const uint32_t sa = smem_u32(stage_sfa(stage)) + lane * 16, sb = smem_u32(stage_sfb(stage)) + lane * 16;
#pragma unroll
                for (int j = 0; j < kMmasPerStage; ++j) {
                    uint32_t *c = r + j * kSfColsPerMma;
                    ld_shared_v4(sa + j * kAtom, c[0], c[1], c[2], c[3]);
                    ld_shared_v4(sb + j * kAtom, c[4], c[5], c[6], c[7]);
                    ld_shared_v4(sb + (kMmasPerStage + j) * kAtom, c[8], c[9], c[10], c[11]);
                }
                const uint32_t dst = lane_base + stage * kSfColsPerStage;
                (void)BI_IN_BOUNDS(kSfCol + (stage + 1) * kSfColsPerStage <= kTmemCols, p.status);
#pragma unroll
                for (int o = 0; o < kSfColsPerStage; o += 16) tmem_st_32x32b_x16(dst + o, r, o);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(ready_leader + stage * 8);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (every CTA)
        // Each warp owns 32 accumulator rows (its lane quarter) x 128 columns.
        // After handing the accumulator back it writes the rounded rows in two
        // 32 x 64 boxes through its own 4 KB staging buffer (128-byte swizzle:
        // 16-byte chunk c of row r sits at chunk c ^ (r % 8)), stored by TMA
        // as whole 128-byte lines.
        const int e = warp - 2 - kSfWarps;
        const int q = warp & 3;
        const int half = e / 4;                               // which 128 columns of the tile
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + half * (kBN / 2);
        const uint32_t box = smem_u32(out_stage + e * kOutBytes);
        if (lane == 0) tma_prefetch_desc(&tmY);
        int it = 0;
        for (int t = cl; t < total; t += ncl, ++it) {
            int mb, nb;
            tile_of(t, mb, nb);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(tfull, it & 1, abort_flag) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            uint32_t packed[kBN / 4];
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c) {
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
            const int row0 = mb * kBM + h * kHalf + q * 32;
            const int col0 = nb * kBN + half * (kBN / 2);
            if (row0 >= p.M || col0 >= p.N) continue;
#pragma unroll
            for (int rd = 0; rd < 2; ++rd) {
                if (lane == 0) bulk_wait_group_read0();       // the previous box has left the buffer
                __syncwarp();
#pragma unroll
                for (int c = 0; c < kOutCols / 8; ++c) {
                    const uint32_t *w = packed + rd * (kOutCols / 2) + c * 4;
                    st_shared_v4(box + lane * 128 + ((c ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, out_stage + e * kOutBytes, col0 + rd * kOutCols, row0);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    grid_dep_launch();                   // the next kernel may start launching on SMs as they free up
    tc_fence_before();
    cluster_sync();                      // no CTA leaves while a peer may still write or signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// Clusters of this kernel that fit on the device at once (queried once per device).
int resident_clusters(int dev, int sms) {
    static std::once_flag once[kMaxDevices];
    static int count[kMaxDevices];
    std::call_once(once[dev], [&] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sms / kClusterCtas * kClusterCtas), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(gemm_nvfp4_kernel), &cfg) !=
                cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = sms / kClusterCtas;
        }
        count[dev] = n;
    });
    return count[dev];
}

}  // namespace

void plan_gemm_nvfp4(int64_t M, int64_t N, int64_t K, int clusters, bi_plan_t *pl) {
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
    pl->grid = static_cast<int32_t>(kClusterCtas * (tiles < clusters ? tiles : clusters));
    pl->reduce_tree = 0;
}

int nvfp4_clusters(int sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return sms / kClusterCtas;
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(gemm_nvfp4_kernel), kSmem, &configured) != BI_OK)
        return sms / kClusterCtas;
    return resident_clusters(dev, sms);
}

bi_status launch_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B, const uint8_t *B_sf,
                            float alpha, void *Y, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    CUtensorMap ta, tb, tsa, tsb, ty;
    // With fewer than 128 rows, each CTA copies only the A rows that can hold
    // data (rounded up to 16); the MMA still multiplies the whole tile and the
    // accumulator rows past M are never stored. Rows never interact, so no
    // stored bit changes.
    const int a_rows = M >= kHalf ? kHalf : static_cast<int>((M + 15) / 16 * 16);
    st = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K / 2, M, K / 2, kBKBytes, a_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
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
    st = make_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, N, M, N * 2, kOutCols, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BI_OK) return st;
    bi_plan_t pl;
    plan_gemm_nvfp4(M, N, K, nvfp4_clusters(info->sm_count), &pl);
    Params p{};
    p.alpha = alpha;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.atoms_per_rowblock = static_cast<int32_t>(K / 64);
    p.stage_tx = kStageBytes - (kHalf - a_rows) * kBKBytes;   // the A box is a_rows high
    p.status = device_status_word();
    return launch_pdl(gemm_nvfp4_kernel, dim3(pl.grid), dim3(kThreads), kSmem, s, ta, tb, tsa, tsb, ty, p);
}

}  // namespace bi
