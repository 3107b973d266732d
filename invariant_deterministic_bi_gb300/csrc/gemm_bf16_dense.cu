// gemm_bf16_dense.cu -- the batch-invariant dense linear layer Y = X W^T
// (bf16 in and out, fp32 accumulation), on CTA pairs (tcgen05 cta_group::2).
//
// Arithmetic, the same for every M and fixed by (N, K) alone:
//   - the K range is cut into S segments of whole 64-wide K steps
//     (S = segments_for(N, K), 1..4; segment s holds steps
//     [s*T/S, (s+1)*T/S) of the T = ceil(K/64) steps);
//   - segment s accumulates its steps in ascending order, from zero, with
//     tcgen05.mma.cta_group::2.kind::f16 (256 x 256 x 16, four per step),
//     giving an fp32 partial P_s of every output element;
//   - Y = bf16_rne( ((P_0 + P_1) + ...) + P_{S-1} ), the partials added in
//     segment order with fp32 additions rounded to nearest even.
// This is a fixed split of the reduction (the pages' batch-invariant GEMM
// keeps one fixed reduction order for all M; here that order includes the
// segments), so no M-dependent split-K, tile shape or stream-K appears.
//
// With S = 1 the layer runs on the lean CTA-pair kernel of gemm_bf16_pair.cu
// (one accumulation, 192 threads, no running sum to hold). With S > 1 two
// schedules of this file's kernel perform exactly these operations:
//   - one pair per 256 x 256 tile (any M, persistent grid): the pair runs
//     the tile's S segments back to back, each into one of two tensor-memory
//     accumulators, and the epilogue warps fold each finished partial into
//     registers (R = P_0, then R = R + P_s) while the next segment runs;
//   - S pairs per tile (M <= 256 and S > 1, one cluster of 2S CTAs per
//     column tile): pair s computes segment s; the running sum passes from
//     each CTA of pair s to the same CTA of pair s + 1 through distributed
//     shared memory (pair s + 1 adds its partial to it), and the last pair
//     rounds and stores. With few
//     rows the tile's K loop is bound by the tensor pipe's fixed cost per
//     step, so this spreads the weight stream over S times more SMs.
// Only which SMs perform the operations, and when, depends on M.
//
// Roles per CTA (384 threads, three warpgroups): warp 0 TMA producer (its
// own 128 rows of A and its half of B per step, both CTAs' copies counted on
// the pair leader's barrier); warp 1 MMA issuer (pair leader only); warps
// 2-3 idle; warps 4-11 epilogue, two per tensor-memory lane quarter, 128
// columns each, storing 32 x 64 boxes through a swizzled staging buffer with
// TMA (rows past M and columns past N are clipped by the tensor map). The
// first warpgroup hands registers to the epilogue warpgroups (setmaxnreg:
// 56 and 224 a thread, the 168 a thread the block is launched with), which
// hold a running sum of 128 fp32 columns a thread.
#include <cuda_bf16.h>

#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kBM = 256;        // pair tile rows (128 per CTA)
constexpr int kHalf = 128;      // rows per CTA of A, and of B
constexpr int kBN = 256;        // pair tile columns = MMA N
constexpr int kBK = 64;
constexpr int kMmaK = 16;
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 4;                    // epilogue warps are 4 .. 11 (warpgroups 1 and 2)
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kRegsLaunch = 168, kRegsLow = 56, kRegsHigh = 224;
static_assert(kRegsLaunch * kThreads >= kRegsLow * 128 + kRegsHigh * 256, "register split fits the launch");
constexpr int kGroupM = 8;      // 8 pair tiles (2048 rows) per raster band
constexpr int kABytes = kHalf * kBK * 2;
constexpr int kBBytes = kHalf * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kOutCols = 64;                    // bf16 columns per output box (128 bytes)
constexpr int kOutBytes = 32 * kOutCols * 2;    // one 32-row box per epilogue warp
constexpr int kColsPerWarp = kBN / 2;           // accumulator columns each epilogue warp owns
constexpr int kBarBytes = 512;
constexpr int kSmem = 1024 + kStages * kStageBytes + kEpiWarps * kOutBytes + kBarBytes;
static_assert(kSmem <= 232448, "shared memory per CTA");
constexpr int kTmemCols = 512;                  // two 256-column accumulators

constexpr int kMinSegmentSteps = 16;            // at least 1024 of K per segment
constexpr int kChainMaxRows = kBM;              // the cluster schedule covers one row tile
// Running sum of one epilogue warp (32 rows x 128 fp32 columns) as it travels
// to the next pair: it lands in that pair's (then idle) operand ring.
constexpr int kSumBytes = 32 * kColsPerWarp * 4;
static_assert(kEpiWarps * kSumBytes <= kStages * kStageBytes, "running sums fit the operand ring");

struct Params {
    int32_t M, N, K;
    int32_t a_bytes;           // A bytes each CTA loads per K step (fewer rows when M < 128)
    int32_t segs;              // S
    int32_t k_steps;           // T
    unsigned *status;
};

__device__ __forceinline__ int seg_begin(int s, int segs, int steps) { return s * steps / segs; }

// ---- cluster-scope synchronisation of the running-sum hand-over
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait with acquire semantics at cluster scope (data written by
// another CTA of the cluster before its release-arrive is visible after it).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, const volatile int *abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}
// Arrive on a barrier of another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Byte offset of 16-byte chunk c (4 columns) of row l in a 32 x 128 fp32
// running sum: rows of 512 bytes, chunks rotated by the row so that the 32
// lanes of a warp (one row each) touch 32 different bank groups.
__device__ __forceinline__ uint32_t sum_off(int l, int c) {
    return static_cast<uint32_t>(l * 512 + (((c ^ l) & 31) << 4));
}

template <bool CHAIN>
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_dense_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmY, const Params p) {
    constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    uint8_t *out_stage = smem + kStages * kStageBytes;    // one staging box per epilogue warp
    uint64_t *full = reinterpret_cast<uint64_t *>(out_stage + kEpiWarps * kOutBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;          // [2] accumulator holds a finished partial
    uint64_t *tempty = tfull + 2;               // [2] accumulator read out (epilogue warps of both CTAs)
    uint64_t *sum_full = tempty + 2;            // [kEpiWarps] running sum from the previous pair has landed
    uint64_t *sum_free = sum_full + kEpiWarps;  // [kEpiWarps] the next pair can take a running sum
    uint64_t *drain = sum_free + kEpiWarps;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    static_assert((2 * kStages + 4 + 2 * kEpiWarps + 1) * 8 + 8 <= kBarBytes, "barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t h = rank & 1u;                       // lane half of the pair's tile
    const uint32_t lead = rank & ~1u;                   // the pair's leader: issues the MMAs
    const uint16_t pair_mask = static_cast<uint16_t>(3u << lead);
    const int csize = CHAIN ? 2 * p.segs : 2;
    const int my_seg = CHAIN ? static_cast<int>(rank >> 1) : 0;
    const int unit = static_cast<int>(blockIdx.x) / csize, nunits = static_cast<int>(gridDim.x) / csize;
    const int num_m = (p.M + kBM - 1) / kBM;
    const int num_n = (p.N + kBN - 1) / kBN;
    const int total = CHAIN ? num_n : num_m * num_n;
    const int seg_lo = CHAIN ? my_seg : 0, seg_hi = CHAIN ? my_seg + 1 : p.segs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * kEpiWarps);
        }
        for (int e = 0; e < kEpiWarps; ++e) {
            mbar_init(&sum_full[e], 1);           // the receiving warp's expect-tx; the bytes come by bulk copy
            mbar_init(&sum_free[e], 1);
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
    tc_fence_before();
    cluster_sync();       // every CTA's barriers exist, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto tile_of = [&](int t, int &mb, int &nb) {
        if (CHAIN) {
            mb = 0;
            nb = t;
            return;
        }
        const int per_group = kGroupM * num_n;
        const int g = t / per_group;
        const int first = g * kGroupM;
        const int gm = min(kGroupM, num_m - first);
        const int local = t - g * per_group;
        mb = first + local % gm;
        nb = local / gm;
    };
    auto give_up = [&]() {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
    };

    if (warp < kEpiWarp0) setmaxnreg_dec<kRegsLow>();
    if (warp == 0) {
        // ------------------------------------------------ TMA producer (every CTA)
        if (lane == 0) {
            const uint32_t full_leader = mapa_shared(smem_u32(full), lead);
            const int kb_lo = seg_begin(seg_lo, p.segs, p.k_steps), kb_hi = seg_begin(seg_hi, p.segs, p.k_steps);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            for (int t = unit; t < total && ok; t += nunits) {
                int mb, nb;
                tile_of(t, mb, nb);
                const int a_row = mb * kBM + static_cast<int>(h) * kHalf;
                const int b_row = nb * kBN + static_cast<int>(h) * kHalf;
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    // debug build: the copy's coordinates lie inside the operands (padded to whole tiles)
                    if (!BI_IN_BOUNDS(kb * kBK < p.K && a_row < num_m * kBM && b_row < num_n * kBN, p.status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (h == 0) mbar_arrive_expect_tx(&full[stage], 2 * (p.a_bytes + kBBytes));
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
                give_up();
                // the leader's full barriers count both CTAs' bytes: waiting on
                // them lets every copy of the pair in flight land
                if (h == 0)
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
            for (int t = unit; t < total && ok; t += nunits) {
                for (int sg = seg_lo; sg < seg_hi && ok; ++sg, ++it) {
                    const int acc = it & 1;
                    const uint32_t acc_phase = (it >> 1) & 1;
                    if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kBN);
                    const int kb_lo = seg_begin(sg, p.segs, p.k_steps), kb_hi = seg_begin(sg + 1, p.segs, p.k_steps);
                    for (int kb = kb_lo; kb < kb_hi; ++kb) {
                        if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(sA + stage * kABytes);
                        const uint32_t b0 = smem_u32(sB + stage * kBBytes);
#pragma unroll
                        for (int k = 0; k < kBK / kMmaK; ++k)
                            mma_bf16_pair(d, sdesc_k_sw128(a0 + k * kMmaK * 2), sdesc_k_sw128(b0 + k * kMmaK * 2),
                                          kIdesc, (kb != kb_lo || k != 0) ? 1u : 0u);
                        tc_commit_pair(&empty[stage], pair_mask);
                        if (++stage == kStages) { stage = 0; phase ^= 1u; }
                    }
                    if (ok) tc_commit_pair(&tfull[acc], pair_mask);
                }
            }
            if (!ok) {
                give_up();
                tc_commit_pair(drain, static_cast<uint16_t>(1u << lead));
                mbar_wait(drain, 0, nullptr);
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        setmaxnreg_inc<kRegsHigh>();
        // ------------------------------------------------ epilogue (every CTA)
        // Warp e owns accumulator rows 32q .. 32q+31 of its CTA (q = warp % 4,
        // the lane quarter it may read) and columns 128*hc .. 128*hc+127.
        const int e = warp - kEpiWarp0;
        const int q = warp & 3;
        const int hc = e >> 2;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), lead);
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(hc * kColsPerWarp);
        uint8_t *box = out_stage + e * kOutBytes;
        if (lane == 0) tma_prefetch_desc(&tmY);
        int it = 0;
        bool ok = true;
        for (int t = unit; t < total && ok; t += nunits) {
            int mb, nb;
            tile_of(t, mb, nb);
            const int row0 = mb * kBM + static_cast<int>(h) * kHalf + q * 32;
            const bool rows = row0 < p.M;                       // warp-uniform: any of its rows exists
            float R[kColsPerWarp];
            for (int sg = seg_lo; sg < seg_hi; ++sg, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                int w = 1;
                if (lane == 0) w = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    if (lane == 0) give_up();
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (rows && BI_IN_BOUNDS(acc * kBN + hc * kColsPerWarp + kColsPerWarp <= kTmemCols, p.status)) {
                    const uint32_t taddr = lane_base + static_cast<uint32_t>(acc * kBN);
#pragma unroll
                    for (int c = 0; c < kColsPerWarp / 16; ++c) {
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(taddr + c * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            R[16 * c + i] = (sg == seg_lo) ? __uint_as_float(r[i])
                                                           : __fadd_rn(R[16 * c + i], __uint_as_float(r[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);   // accumulator may be reused
            }
            if (!ok) break;
            if (CHAIN) {
                // the running sum moves pair to pair in segment order, each CTA
                // to the CTA holding the same rows in the next pair, through the
                // rows' area of the receiver's operand ring (idle once its MMAs
                // have completed): rows of 512 bytes, one bulk copy per warp
                if (!rows) continue;
                const int nrows = min(32, p.M - row0);
                const uint32_t bytes = static_cast<uint32_t>(nrows) * 512u;
                uint8_t *area = smem + e * kSumBytes;
                // debug build: the running sum stays inside the operand ring, and the pairs of the chain exist
                if (!BI_IN_BOUNDS(e * kSumBytes + static_cast<int>(bytes) <= kStages * kStageBytes &&
                                      (my_seg == 0 || rank >= 2) && (my_seg == p.segs - 1 || static_cast<int>(rank) + 2 < csize),
                                  p.status))
                    continue;
                if (my_seg > 0) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sum_full[e], bytes);
                        mbar_arrive_release_cluster(mapa_shared(smem_u32(&sum_free[e]), rank - 2));
                    }
                    int w = 1;
                    if (lane == 0) w = mbar_wait(&sum_full[e], 0, abort_flag) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, w, 0)) {
                        if (lane == 0) give_up();
                        break;
                    }
                    if (lane < nrows) {
                        const uint32_t in = smem_u32(area);
#pragma unroll
                        for (int c = 0; c < kColsPerWarp / 4; ++c) {
                            uint32_t a, b, cc, d;
                            ld_shared_v4(in + sum_off(lane, c), a, b, cc, d);
                            // earlier segments first: (P_0 + ... + P_{s-1}) + P_s
                            R[4 * c + 0] = __fadd_rn(__uint_as_float(a), R[4 * c + 0]);
                            R[4 * c + 1] = __fadd_rn(__uint_as_float(b), R[4 * c + 1]);
                            R[4 * c + 2] = __fadd_rn(__uint_as_float(cc), R[4 * c + 2]);
                            R[4 * c + 3] = __fadd_rn(__uint_as_float(d), R[4 * c + 3]);
                        }
                    }
                }
                if (my_seg < p.segs - 1) {
                    if (lane < nrows) {
                        const uint32_t out = smem_u32(area);
#pragma unroll
                        for (int c = 0; c < kColsPerWarp / 4; ++c)
                            st_shared_v4(out + sum_off(lane, c), __float_as_uint(R[4 * c]), __float_as_uint(R[4 * c + 1]),
                                         __float_as_uint(R[4 * c + 2]), __float_as_uint(R[4 * c + 3]));
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    int w = 1;
                    if (lane == 0) {
                        w = mbar_wait_cluster(&sum_free[e], 0, abort_flag) ? 1 : 0;
                        if (w)
                            bulk_copy_to_cluster(mapa_shared(smem_u32(area), rank + 2), area, bytes,
                                                 mapa_shared(smem_u32(&sum_full[e]), rank + 2));
                    }
                    if (!__shfl_sync(0xffffffffu, w, 0)) {
                        if (lane == 0) give_up();
                        break;
                    }
                    continue;                                  // the last pair stores
                }
            }
            if (!rows) continue;
            // round to bf16 and store two 32 x 64 boxes (128-byte swizzle: 16-byte
            // chunk c of row r at chunk c ^ (r % 8))
            const int col0 = nb * kBN + hc * kColsPerWarp;
#pragma unroll
            for (int bx = 0; bx < kColsPerWarp / kOutCols; ++bx) {
                if (col0 + bx * kOutCols >= p.N) break;
                if (lane == 0) bulk_wait_group_read0();        // the previous box has left the buffer
                __syncwarp();
                const uint32_t sb = smem_u32(box) + lane * 128;
#pragma unroll
                for (int c = 0; c < kOutCols / 8; ++c) {
                    const float *v = R + bx * kOutCols + c * 8;
                    st_shared_v4(sb + ((c ^ (lane & 7)) << 4),
                                 pack_bf16x2(__float_as_uint(v[0]), __float_as_uint(v[1])),
                                 pack_bf16x2(__float_as_uint(v[2]), __float_as_uint(v[3])),
                                 pack_bf16x2(__float_as_uint(v[4]), __float_as_uint(v[5])),
                                 pack_bf16x2(__float_as_uint(v[6]), __float_as_uint(v[7])));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, box, col0 + bx * kOutCols, row0);
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    grid_dep_launch();                   // the next kernel may start launching on SMs as they free up
    tc_fence_before();
    cluster_sync();                      // no CTA leaves while a peer may still write into it or signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

bi_status launch_cluster(void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, Params), int csize, int grid,
                         cudaStream_t s, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ty,
                         const Params &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, ty, p) == cudaSuccess) return BI_OK;
    cudaGetLastError();   // reported here; do not leave it for a later, unrelated check
    return BI_ERR_CUDA;
}

}  // namespace

// Segments of the K reduction for an N x K layer, from (N, K) alone (not M,
// not the device): S in 1..4, each segment at least 16 steps of 64. The
// choice minimises a cost, in K steps, of one row tile of the layer on a
// 152-SM GB300: with S = 1, ceil(tiles_n / 76 pairs) rounds of T + 8 steps
// (the 8 stand for set-up and epilogue); with S > 1, ceil(tiles_n / c_S)
// rounds of ceil(T / S) + 8 + 6 (S - 1) steps, where c_S is the number of
// 2S-CTA clusters of this kernel resident at once on that GPU (measured: 36
// of 4 CTAs, 23 of 6, 15 of 8) and 6 steps stand for each hand-over of the
// running sum. S > 1 is taken only when it costs at most 3/4 of S = 1, since
// at large M it adds work (the epilogue folds every segment) for no gain.
int segments_for(int64_t N, int64_t K) {
    const int64_t T = (K + kBK - 1) / kBK;
    const int64_t tiles_n = (N + kBN - 1) / kBN;
    const int64_t cost1 = ((tiles_n + 75) / 76) * (T + 8);
    const int64_t cap[5] = {0, 0, 36, 23, 15};
    int best = 1;
    int64_t best_cost = cost1;
    for (int S = 2; S <= 4; ++S) {
        if (T / S < kMinSegmentSteps) break;
        const int64_t cost = ((tiles_n + cap[S] - 1) / cap[S]) * ((T + S - 1) / S + 8 + 6 * (S - 1));
        if (4 * cost <= 3 * cost1 && cost < best_cost) {
            best = S;
            best_cost = cost;
        }
    }
    return best;
}

// The cluster schedule (S pairs per tile) is used when the rows fit one row
// tile and there is more than one segment.
static bool use_chain(int64_t M, int segs) { return segs > 1 && M <= kChainMaxRows; }

void plan_gemm_bf16(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *pl) {
    if (segments_for(N, K) == 1) {      // one segment: the lean CTA-pair kernel of gemm_bf16_pair.cu
        plan_gemm_bf16_one_segment(M, N, K, sms, pl);
        return;
    }
    pl->op = BI_OP_GEMM_BF16;
    pl->block_m = kBM; pl->block_n = kBN; pl->block_k = kBK;
    pl->mma_m = kBM; pl->mma_n = kBN; pl->mma_k = kMmaK;
    pl->k_steps = static_cast<int32_t>((K + kBK - 1) / kBK);
    pl->split_k = segments_for(N, K);
    pl->stages = kStages;
    pl->threads = kThreads;
    pl->smem_bytes = kSmem;
    pl->tiles_m = (M + kBM - 1) / kBM;
    pl->tiles_n = (N + kBN - 1) / kBN;
    if (use_chain(M, pl->split_k)) {
        pl->grid = static_cast<int32_t>(pl->tiles_n * 2 * pl->split_k);   // one cluster per column tile
    } else {
        const int64_t tiles = pl->tiles_m * pl->tiles_n;
        const int64_t pairs = sms / 2;
        pl->grid = static_cast<int32_t>(2 * (tiles < pairs ? tiles : pairs));
    }
    pl->reduce_tree = 0;
}

bi_status launch_gemm_bf16(const void *X, int64_t ldx, const void *W, int64_t ldw, void *Y, int64_t ldy,
                           int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    if (segments_for(N, K) == 1) return launch_gemm_bf16_one_segment(X, ldx, W, ldw, Y, ldy, M, N, K, s);
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
    plan_gemm_bf16(M, N, K, info->sm_count, &pl);
    Params p{};
    p.a_bytes = a_rows * kBK * 2;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.segs = pl.split_k;
    p.k_steps = pl.k_steps;
    p.status = device_status_word();
    const bool chain = use_chain(M, p.segs);
    auto kern = chain ? gemm_bf16_dense_kernel<true> : gemm_bf16_dense_kernel<false>;
    static unsigned long long configured[2] = {0, 0};
    if (ensure_smem_attr(reinterpret_cast<const void *>(kern), kSmem, &configured[chain ? 1 : 0]) != BI_OK)
        return BI_ERR_CUDA;
    return launch_cluster(kern, chain ? 2 * p.segs : 2, pl.grid, s, ta, tb, ty, p);
}

}  // namespace bi
