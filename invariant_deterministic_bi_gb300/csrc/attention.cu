// attention.cu -- batch-invariant decode attention over a paged KV cache.
//
// Batch-invariant attention is on the vLLM tracking issue's TODO list
// (FlashInfer, TRITON_MLA, FLASHINFER_MLA support) and the vllm-ascend guide
// lists batch-invariant attention operators. Split-KV ("flash decoding")
// kernels usually pick the number of KV splits from the batch size to fill the
// GPU; that makes a sequence's reduction order depend on the batch. Here the
// split is fixed: a sequence's KV is cut into chunks of kChunk = 128 tokens by
// position alone, every chunk is reduced by one CTA in a fixed order, and the
// chunk results are merged in chunk order. Nothing a sequence sees depends on
// the other sequences in the batch.
//
// Step 1, per (sequence, KV head, chunk of kChunk = 128 tokens) item, head_dim
//   128, the G = Hq/Hkv query heads of the KV head together (GQA), computed
//   by a persistent kernel (one CTA per SM walking the items; details at
//   attn_split_kernel):
//   - the chunk's K and V rows arrive in shared memory by TMA (one box per
//     cache block; blocks outside the cache arrive as zeros and score -inf);
//   - scores on the tensor cores (mma.sync m16n8k16, bf16 operands, fp32
//     accumulation): the G q rows (zero rows up to 16) times K^T, every
//     8-token n-tile's chain of MMAs in ascending 16-dimension steps;
//     s = scale * q.k;
//   - per head (one warp): m = max s (exact), p = exp(s - m), l = sum p
//     (lane L sums tokens L, L + 32, L + 64, L + 96 in turn, then a
//     butterfly over lanes xor 16, 8, 4, 2, 1);
//   - values on the tensor cores: p (as bf16 hi + lo, two MMAs per step, 16
//     significant bits) times V, every 8-dimension tile's chain in
//     ascending 16-token steps, hi before lo;
//   - writes fp32 (m, l, o[0..127]) per head and chunk to the workspace.
//   The MMA shapes and step orders are the same for every chunk of every
//   batch, and which warp or CTA computes a tile changes nothing, so the
//   per-chunk results do not depend on the batch either.
// Step 2, one CTA per (sequence, query head): the chunk results are merged
//   in chunk order by merge_factors() / merge_value() below (running maximum
//   m, with the running o and l rescaled by e^{m - m'} and the chunk's by
//   e^{m_c - m'}), and o / l is rounded to bf16.
//
// Extend (prefill) attention, attn_extend_kernel: the new query tokens of a
// sequence attend causally to its cache. Token i at position p sees tokens
// 0..p, so its result is defined as the decode result of the sequence cut
// after p: the same 128-token chunks by position, the same per-chunk
// arithmetic (the same MMA chains, max, e^(s-m), the same sum order, p.V with
// p as bf16 hi + lo) and the same chunk-order merge. A token's output is
// therefore the same bits whether it is decoded alone, prefilled at once,
// prefilled in chunks of any size, or batched with other sequences. One CTA
// per (sequence, KV head, 128 query rows = 128/G tokens x G heads) walks the
// chunks in order; each warp keeps 16 rows' scores, exponentials and running
// (m, l, o) in registers.
#include <cuda_bf16.h>

#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 128;                    // tokens per chunk: fixed, by position
constexpr int kThreads = 256;                  // split kernel
constexpr int kCombineThreads = 128;           // one thread per output dimension
constexpr int kRowBytes = kD * 2;              // one token's K (or V) row of one KV head
constexpr int kTileBytes = kChunk * kRowBytes; // 32 KB


// 16-byte global -> shared copy; src_bytes = 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// D += A B on the tensor cores, one warp: A 16x16 bf16 (row-major fragment
// a0..a3), B 16x8 bf16 (column fragment b0, b1), D 16x8 fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8x8 bf16 matrices from shared memory, transposed (lanes 8i..8i+7 give
// the 16-byte rows of matrix i).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                                  uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// Four 8x8 bf16 matrices from shared memory (lanes 8i..8i+7 give the 16-byte
// rows of matrix i); lane (g, c) receives row g, columns 2c and 2c+1 of each.
__device__ __forceinline__ void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// (p0, p1) = hi + lo, hi and lo packed bf16 pairs (round to nearest even);
// hi + lo carries 16 significant bits of each p.
__device__ __forceinline__ void split_bf16x2(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(__float_as_uint(p0), __float_as_uint(p1));
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
    lo = pack_bf16x2(__float_as_uint(p0 - h0), __float_as_uint(p1 - h1));
}

// Merge one chunk's (m_c, l_c, o_c) into the running (m, l, o) of a query
// row, in chunk order: m' = max(m, m_c); o = o e^{m - m'} + o_c e^{m_c - m'},
// l likewise (the first chunk finds m = -inf, l = o = 0). Decode and extend
// attention both merge through this one definition.
__device__ __forceinline__ void merge_factors(float m, float m_c, float &m_new, float &alpha, float &beta) {
    m_new = fmaxf(m, m_c);
    alpha = expf(__fsub_rn(m, m_new));
    beta = expf(__fsub_rn(m_c, m_new));
}
__device__ __forceinline__ float merge_value(float run, float chunk, float alpha, float beta) {
    return __fmaf_rn(chunk, beta, __fmul_rn(run, alpha));
}

struct AttnParams {
    const uint16_t *Q;       // [B][Hq][D]
    const uint16_t *K;       // [blocks][bs][Hkv][D]
    const uint16_t *V;
    const int32_t *table;    // [B][max_blocks]
    const int32_t *lens;     // [B]
    float *ws;               // [B][Hq][chunks][kD + 2]
    uint16_t *O;             // [B][Hq][D]
    int64_t num_blocks, batch;
    int32_t max_blocks, Hq, Hkv, bs, chunks, max_len;
    int32_t box_rows;        // tokens per TMA box of the decode loader; 0: per-row copies
    float scale;
    unsigned *status;
};

// A read-only load issued where it stands (the table is not written while a
// kernel of this file runs).
__device__ __forceinline__ int32_t ld_nc_s32(const int32_t *ptr) {
    int32_t v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

__device__ __forceinline__ bool seq_ok(const AttnParams &p, int64_t b, int &L) {
    L = p.lens[b];
    return L >= 1 && L <= p.max_len && L <= static_cast<int64_t>(p.max_blocks) * p.bs;
}

// Step 1 runs persistently: one CTA per SM walks the (sequence, KV head,
// chunk) items blockIdx.x, blockIdx.x + gridDim.x, ... (which CTA computes an
// item changes no arithmetic). A loading warp keeps up to kSlots chunks in
// flight: per item it resolves the chunk's block-table entries and loads the
// chunk's K and V rows of KV head g with TMA, one box per cache block (a 4-D
// tensor map over [blocks][block size][KV heads][128], two 64-dimension
// halves per box, 128-byte swizzle), plus the G q rows by a bulk copy, all
// counted on the slot's "full" barrier. Block sizes that boxes cannot tile
// (not a multiple of 128 and not 8, 16, 32 or 64) take 16-byte cp.async
// copies per row instead. Blocks outside the cache arrive as zeros and their
// tokens score -inf. Eight consumer warps, in NG groups, compute the chunks
// and hand each slot back through its "empty" barrier.
//
// Two shapes of the kernel, the same arithmetic per item:
//   - many items: SLOTS = 3 ring slots, NG = 2 groups of four warps on
//     alternate items (two items in compute while up to three load), one CTA
//     per SM;
//   - few items (at most two CTAs' worth per SM): SLOTS = 1, NG = 1, one item
//     per CTA on all eight warps, two CTAs per SM; the V rows are counted on
//     a second "full" barrier, so that the scores start as soon as K and q
//     have landed.
constexpr int kHalfTile = kChunk * 128;                  // one 64-dimension half of a K or V tile (swizzled)
constexpr int kSlotBytes = 4 * kHalfTile + 8 * kRowBytes; // K, V, up to 8 q rows
constexpr int kDecConsumers = kThreads / 32;             // 8 warps
constexpr int kDecSStride = kChunk + 8;                 // scores of one head (padded)
constexpr int kDecSFloats = 8 * kDecSStride;             // one score buffer: up to 8 heads
template <int SLOTS>
constexpr int dec_threads() { return kThreads + 32 * SLOTS; }   // + one loading warp per slot
template <int SLOTS, int NG>
constexpr int dec_smem() {
    return 1024 + SLOTS * kSlotBytes + 2 * NG * kDecSFloats * 4 + SLOTS * kChunk + (2 * NG + 1) * SLOTS * 8 + 16;
}
static_assert(kSlotBytes % 1024 == 0, "slot alignment (128-byte swizzle atoms)");
static_assert(2 * dec_smem<1, 1>() <= 232448, "two few-item CTAs per SM");

// Byte offset of 16-byte piece x (0..15) of token row t in a swizzled K or V tile.
__device__ __forceinline__ int kv_piece(int t, int x) {
    return (x >> 3) * kHalfTile + t * 128 + (((x & 7) ^ (t & 7)) << 4);
}

// bar.sync on the named barrier (1 + grp) of consumer group grp's GW warps
template <int GW>
__device__ __forceinline__ void group_sync(int grp) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(32 * GW) : "memory");
}
// the same barrier with an OR vote over the group's threads
template <int GW>
__device__ __forceinline__ bool group_sync_or(int grp, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(1 + grp), "n"(32 * GW)
        : "memory");
    return r != 0;
}

template <int G, int kSlots, int NG>
__global__ void __launch_bounds__(dec_threads<kSlots>(), kSlots == 1 ? 2 : 1)
attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const AttnParams p) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *S0 = reinterpret_cast<float *>(smem + kSlots * kSlotBytes);     // [group][2][G][kDecSStride] scores
    uint8_t *valid = reinterpret_cast<uint8_t *>(S0 + 2 * NG * kDecSFloats); // [kSlots][kChunk]: row has K/V
    // Barriers. Every waiter waits only for the phase right after one it has
    // seen complete (a parity wait cannot tell a phase from the one two
    // later): slot s is filled by one loading warp in item order, so one
    // "empty" barrier per slot serves it; the items of a slot alternate
    // between the consumer groups, so each (slot, group) has its own "full"
    // barrier, whose phases are that group's items on that slot in order.
    // With one item per CTA (kSlots = 1) the V rows have a "full" barrier of
    // their own (fullV); the ring counts them with the K rows.
    constexpr bool kSplitKV = kSlots == 1;
    uint64_t *full = reinterpret_cast<uint64_t *>(valid + kSlots * kChunk);   // [kSlots][NG]
    uint64_t *fullV = full + kSlots * NG;                                     // [kSlots][NG], kSplitKV only
    uint64_t *empty = fullV + kSlots * NG;                                    // [kSlots]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kSlots);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kSlots * NG; ++s) {
            mbar_init(&full[s], p.box_rows > 0 ? 32 : 64);
            mbar_init(&fullV[s], p.box_rows > 0 ? 32 : 64);
        }
        for (int s = 0; s < kSlots; ++s) mbar_init(&empty[s], kDecConsumers / NG);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int64_t items = p.batch * p.Hkv * static_cast<int64_t>(p.chunks);
    // item -> (sequence b, KV head g, chunk c) and the tokens n of the chunk;
    // false when the chunk is past the sequence (or the sequence is invalid)
    auto item = [&](int64_t it, int64_t &b, int &g, int &c, int &n) {
        g = static_cast<int>(it % p.Hkv);               // KV head fastest: the heads of one
        const int64_t r = it / p.Hkv;                    // cache block are read together
        c = static_cast<int>(r % p.chunks);
        b = r / p.chunks;
        int L;
        if (!seq_ok(p, b, L)) {
            if (warp == kDecConsumers && lane == 0 && c == 0 && g == 0) atomicOr(p.status, kDevBadOffsets);   // loader 0
            return false;
        }
        n = min(kChunk, L - c * kChunk);
        return n > 0;
    };

    if (warp >= kDecConsumers) {
        // ---- loading warps: warp lw fills slot lw with items lw, lw + 3, ... (a
        // table read and the copies' issue per item), so three items are
        // prepared at a time
        const int lw = warp - kDecConsumers;
        if (lane == 0 && p.box_rows > 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        // K and V rows are read once: evict them from L2 first, so that the
        // chunk partials the combine step reads stay there
        const uint64_t kv_policy = l2_policy_evict_first();
        int k = 0, last = -1;
        for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
            // the item's block-table entries (boxes: lane i < kChunk / box_rows
            // reads box i's) are requested before its sequence length is
            // known, so the two reads overlap instead of following each other
            int32_t spec_blk = -1;
            if (p.box_rows > 0) {
                const int64_t r = it / p.Hkv;
                const int64_t bb = r / p.chunks;
                const int64_t bi = ((r % p.chunks) * kChunk + lane * p.box_rows) / p.bs;
                if (lane < kChunk / p.box_rows && bb < p.batch && bi < p.max_blocks)
                    spec_blk = ld_nc_s32(p.table + bb * p.max_blocks + bi);
            }
            int64_t b;
            int g, c, n;
            if (!item(it, b, g, c, n)) continue;
            if (k % kSlots != lw) {
                ++k;
                continue;
            }
            // the block-table reads first: they do not touch the slot
            const int j0 = c * kChunk;
            int64_t off[kChunk / 32];                 // per-row copies: element offset of each row, -1: none
            bool ok_row[kChunk / 32];                 // the row's block is inside the cache
            int32_t box_blk = -1;                     // boxes: lane i < nbox holds box i's block
            const int nbox = p.box_rows > 0 ? (n + p.box_rows - 1) / p.box_rows : 0;
            if (p.box_rows > 0) {
                if (lane < nbox) {
                    box_blk = spec_blk;            // p.table[b][(j0 + lane * box_rows) / bs]
                    if (box_blk < 0 || box_blk >= p.num_blocks) atomicOr(p.status, kDevBadOffsets);
                }
#pragma unroll
                for (int i = 0; i < kChunk / 32; ++i) {
                    const int t = lane + 32 * i;
                    const int32_t blk = __shfl_sync(0xffffffffu, box_blk, t / p.box_rows);
                    ok_row[i] = t < n && blk >= 0 && blk < p.num_blocks;
                    off[i] = -1;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kChunk / 32; ++i) {
                    const int t = lane + 32 * i;
                    off[i] = -1;
                    if (t < n) {
                        const int j = j0 + t;
                        const int64_t blk = p.table[b * p.max_blocks + j / p.bs];
                        if (blk >= 0 && blk < p.num_blocks)
                            off[i] = ((blk * p.bs + j % p.bs) * p.Hkv + g) * kD;
                        else
                            atomicOr(p.status, kDevBadOffsets);
                    }
                    ok_row[i] = off[i] >= 0;
                }
            }
            const int slot = k % kSlots;
            uint64_t *fb = &full[slot * NG + k % NG];   // the consuming group's barrier for this slot
            uint64_t *fbv = kSplitKV ? &fullV[slot * NG + k % NG] : fb;   // the one counting the V rows
            if (k >= kSlots && !mbar_wait(&empty[slot], ((k / kSlots) - 1) & 1, abort_flag)) {
                if (lane == 0) {
                    atomicOr(p.status, kDevTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            uint8_t *Ks = smem + slot * kSlotBytes;
            uint8_t *Vs = Ks + 2 * kHalfTile;
            uint8_t *qs = Vs + 2 * kHalfTile;
#pragma unroll
            for (int i = 0; i < kChunk / 32; ++i) valid[slot * kChunk + lane + 32 * i] = ok_row[i];
            const uint16_t *qsrc = p.Q + (b * p.Hq + g * G) * kD;
            if (p.box_rows > 0) {
                // one box per cache block (box_rows tokens), both halves
                const int kv_bytes = nbox * p.box_rows * 2 * 128;   // the K rows, or the V rows
                const int tok = (j0 + lane * p.box_rows) % p.bs;
                // V rows no box reaches (a chunk past the sequence's end) become
                // zero, so that p = 0 meets finite values there; each lane's
                // arrival on the barrier counting the V rows releases its zeros
                auto zero_v_tail = [&] {
                    for (int r = nbox * p.box_rows + lane; r < kChunk; r += 32) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint4 *v = reinterpret_cast<uint4 *>(Vs + half * kHalfTile + r * 128);
#pragma unroll
                            for (int x = 0; x < 8; ++x) v[x] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();         // before later bulk copies into these rows
                    __syncwarp();
                };
                if (!kSplitKV) zero_v_tail();
                __syncwarp();
                // each lane's arrival releases its shared-memory writes; lane 0
                // also sets the bytes to expect, before any copy is issued
                if (lane == 0)
                    mbar_arrive_expect_tx(fb, (kSplitKV ? 1 : 2) * kv_bytes + G * kRowBytes);
                else
                    mbar_arrive(fb);
                __syncwarp();
                if (kSplitKV) {
                    // q and K first: the scores need them before p.V needs V
                    if (lane == 0) bulk_load(qs, qsrc, G * kRowBytes, fb);
                    if (lane < nbox) {                // a block outside the cache arrives as zeros
#pragma unroll
                        for (int half = 0; half < 2; ++half)
                            tma_load_4d_hint(Ks + half * kHalfTile + lane * p.box_rows * 128, &tmK, fb, half * 64, g,
                                             tok, box_blk, kv_policy);
                    }
                    zero_v_tail();
                    if (lane == 0)
                        mbar_arrive_expect_tx(fbv, kv_bytes);
                    else
                        mbar_arrive(fbv);
                    __syncwarp();
                    if (lane < nbox) {
#pragma unroll
                        for (int half = 0; half < 2; ++half)
                            tma_load_4d_hint(Vs + half * kHalfTile + lane * p.box_rows * 128, &tmV, fbv, half * 64, g,
                                             tok, box_blk, kv_policy);
                    }
                } else {
                    // the ring consumes a slot whole: K and V boxes in turn, then q
                    if (lane < nbox) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int dst = half * kHalfTile + lane * p.box_rows * 128;
                            tma_load_4d_hint(Ks + dst, &tmK, fb, half * 64, g, tok, box_blk, kv_policy);
                            tma_load_4d_hint(Vs + dst, &tmV, fb, half * 64, g, tok, box_blk, kv_policy);
                        }
                    }
                    if (lane == 0) bulk_load(qs, qsrc, G * kRowBytes, fb);
                }
            } else {
                // 16-byte copies per row (rows without K/V zero-filled); each lane
                // arrives twice: now, and once its copies have landed (both on
                // the V rows' barrier too, when it has its own)
#pragma unroll
                for (int i = 0; i < kChunk / 32; ++i) {
                    const int t = lane + 32 * i;
                    for (int x = 0; x < kRowBytes / 16; ++x) {
                        const uint32_t so = kv_piece(t, x);
                        cp_async_16(smem_u32(Ks) + so, off[i] >= 0 ? p.K + off[i] + x * 8 : p.K, off[i] >= 0 ? 16u : 0u);
                        cp_async_16(smem_u32(Vs) + so, off[i] >= 0 ? p.V + off[i] + x * 8 : p.V, off[i] >= 0 ? 16u : 0u);
                    }
                }
                for (int x = lane; x < G * kRowBytes / 16; x += 32) cp_async_16(smem_u32(qs) + x * 16, qsrc + x * 8, 16u);
                mbar_arrive(fb);                      // releases this lane's row flags
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(fb)) : "memory");
                if (kSplitKV) {
                    mbar_arrive(fbv);
                    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(fbv)) : "memory");
                }
            }
            last = k;
            ++k;
        }
        // the copies of this warp's last item must land before the CTA exits
        // (the consumers normally waited for them already; every earlier item
        // of the slot was consumed before the slot was filled again)
        if (last >= 0) {
            mbar_wait(&full[(last % kSlots) * NG + last % NG], (last / (kSlots * NG)) & 1, nullptr);
            if (kSplitKV) mbar_wait(&fullV[(last % kSlots) * NG + last % NG], (last / (kSlots * NG)) & 1, nullptr);
        }
        return;
    }

    // ---- consumer warps 0..7: group grp (warps GW grp .. GW grp + GW - 1)
    // computes the items k with k % NG == grp; how the warps share an item
    // changes no arithmetic
    constexpr int GW = kDecConsumers / NG;                // warps per group
    constexpr int NT = kChunk / 8 / GW;                   // score n-tiles per warp
    constexpr int DW = kD / GW;                           // value dimensions per warp
    const int grp = warp / GW, gw = warp % GW;
    const int gq = lane >> 2, cq = lane & 3;              // fragment row group, column pair
    const int64_t ws_head = static_cast<int64_t>(p.chunks) * (kD + 2);   // next query head's record
    int k = 0;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        int64_t b;
        int g, c, n;
        if (!item(it, b, g, c, n)) continue;
        if (k % NG != grp) {
            ++k;
            continue;
        }
        const int slot = k % kSlots;
        const bool ok = mbar_wait(&full[slot * NG + grp], (k / (kSlots * NG)) & 1, abort_flag);
        if (group_sync_or<GW>(grp, !ok)) {                    // the group's warps stop together
            if (gw == 0 && lane == 0) {
                atomicOr(p.status, kDevTimeout);
                *abort_flag = 1;
            }
            break;
        }
        const uint8_t *Ks = smem + slot * kSlotBytes;
        const uint8_t *Vs = Ks + 2 * kHalfTile;
        const uint16_t *qb = reinterpret_cast<const uint16_t *>(Vs + 2 * kHalfTile);
        const uint8_t *vrow = valid + slot * kChunk;
        float *S = S0 + (grp * 2 + ((k / NG) & 1)) * kDecSFloats;
        float *wsh = p.ws + ((b * p.Hq + g * G) * p.chunks + c) * static_cast<int64_t>(kD + 2);
        if (!BI_IN_BOUNDS(b < p.batch && c < p.chunks, p.status)) break;

        // scores S[h][t] = q_h . k_t on the tensor cores: A = q (rows = the G
        // heads, zero beyond), B = K^T; warp gw of the group takes tokens
        // 8 NT gw .. 8 NT gw + 8 NT - 1, K ascending in 16-dimension steps
        {
            uint32_t qa[kD / 16][2];
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                qa[ks][0] = gq < G ? *reinterpret_cast<const uint32_t *>(qb + gq * kD + 16 * ks + 2 * cq) : 0u;
                qa[ks][1] = gq < G ? *reinterpret_cast<const uint32_t *>(qb + gq * kD + 16 * ks + 8 + 2 * cq) : 0u;
            }
            // the NT n-tiles' chains interleaved, each in ascending dimension order
            float acc[NT][4] = {};
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                uint32_t bf[NT][2];
#pragma unroll
                for (int nb = 0; nb < NT; ++nb) {
                    const int t = gw * 8 * NT + nb * 8 + gq;   // the K row of this lane's B fragment
                    bf[nb][0] = *reinterpret_cast<const uint32_t *>(Ks + cq * 4 + kv_piece(t, 2 * ks));
                    bf[nb][1] = *reinterpret_cast<const uint32_t *>(Ks + cq * 4 + kv_piece(t, 2 * ks + 1));
                }
#pragma unroll
                for (int nb = 0; nb < NT; ++nb) mma_16816(acc[nb], qa[ks][0], 0u, qa[ks][1], 0u, bf[nb][0], bf[nb][1]);
            }
            if (gq < G) {
#pragma unroll
                for (int nb = 0; nb < NT; ++nb)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tt = gw * 8 * NT + nb * 8 + 2 * cq + e;
                        if (tt < n) S[gq * kDecSStride + tt] = vrow[tt] ? __fmul_rn(acc[nb][e], p.scale) : -INFINITY;
                    }
            }
        }
        group_sync<GW>(grp);

        // per head: max, exponentials, sum (head h on warp h % GW); (m, l) to the workspace
        for (int h = gw; h < G; h += GW) {
            float m = -INFINITY;
            const float *Sh = S + h * kDecSStride;
            for (int t = lane; t < n; t += 32) m = fmaxf(m, Sh[t]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float l = 0.0f;
            for (int t = lane; t < n; t += 32) {
                const float e = expf(Sh[t] - m);
                S[h * kDecSStride + t] = e;
                l += e;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) {
                wsh[h * ws_head] = m;
                wsh[h * ws_head + 1] = l;
            }
        }
        if (kSplitKV) {
            const bool ok_v = mbar_wait(&fullV[slot * NG + grp], (k / (kSlots * NG)) & 1, abort_flag);
            if (group_sync_or<GW>(grp, !ok_v)) {              // the V rows did not land
                if (gw == 0 && lane == 0) {
                    atomicOr(p.status, kDevTimeout);
                    *abort_flag = 1;
                }
                break;
            }
        } else {
            group_sync<GW>(grp);
        }

        // values O[h][d] = sum_t p_t v_t[d] on the tensor cores: A = p (rows =
        // the G heads; p = hi + lo, two bf16 MMAs per step; zero past the
        // chunk's tokens), B = V read transposed by ldmatrix; warp gw takes
        // dimensions DW gw .. DW gw + DW - 1, tokens ascending in 16-token steps
        {
            const int d0 = gw * DW;
            const int mi = lane >> 3, mr = lane & 7;      // ldmatrix: matrix, row
            float acc[DW / 8][4] = {};
            // p of every step first (independent loads), then the MMA chains
            uint32_t ph[kChunk / 16][2], pl[kChunk / 16][2];
#pragma unroll
            for (int ks = 0; ks < kChunk / 16; ++ks) {
                ph[ks][0] = ph[ks][1] = pl[ks][0] = pl[ks][1] = 0u;
                if (gq < G) {
                    const int t0 = ks * 16 + 2 * cq, t2 = t0 + 8;
                    const float *Sq = S + gq * kDecSStride;
                    const float p00 = t0 < n ? Sq[t0] : 0.0f;
                    const float p01 = t0 + 1 < n ? Sq[t0 + 1] : 0.0f;
                    const float p20 = t2 < n ? Sq[t2] : 0.0f;
                    const float p21 = t2 + 1 < n ? Sq[t2 + 1] : 0.0f;
                    split_bf16x2(p00, p01, ph[ks][0], pl[ks][0]);
                    split_bf16x2(p20, p21, ph[ks][1], pl[ks][1]);
                }
            }
#pragma unroll
            for (int ks = 0; ks < kChunk / 16; ++ks) {
                const int k0 = ks * 16;
                const uint32_t ph0 = ph[ks][0], ph2 = ph[ks][1], pl0 = pl[ks][0], pl2 = pl[ks][1];
                const int tok = k0 + (mi & 1) * 8 + mr;
                uint32_t v[DW / 16][4];
#pragma unroll
                for (int hf = 0; hf < DW / 16; ++hf) {    // 16 dimensions per ldmatrix
                    const int piece = ((d0 + 16 * hf) >> 3) + (mi >> 1);
                    ldmatrix_x4_trans(v[hf][0], v[hf][1], v[hf][2], v[hf][3], smem_u32(Vs + kv_piece(tok, piece)));
                }
                // each accumulator takes hi, then lo
#pragma unroll
                for (int hf = 0; hf < DW / 16; ++hf) {
                    mma_16816(acc[2 * hf], ph0, 0u, ph2, 0u, v[hf][0], v[hf][1]);
                    mma_16816(acc[2 * hf + 1], ph0, 0u, ph2, 0u, v[hf][2], v[hf][3]);
                }
#pragma unroll
                for (int hf = 0; hf < DW / 16; ++hf) {
                    mma_16816(acc[2 * hf], pl0, 0u, pl2, 0u, v[hf][0], v[hf][1]);
                    mma_16816(acc[2 * hf + 1], pl0, 0u, pl2, 0u, v[hf][2], v[hf][3]);
                }
            }
            if (gq < G) {
                float *w = wsh + gq * ws_head + 2 + d0 + 2 * cq;
#pragma unroll
                for (int nb = 0; nb < DW / 8; ++nb)
                    *reinterpret_cast<float2 *>(w + nb * 8) = make_float2(acc[nb][0], acc[nb][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);         // this warp is done with the slot
        ++k;
    }
}

__global__ void __launch_bounds__(kCombineThreads)
attn_combine_kernel(const AttnParams p) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    // Chunks in tiles of 32. Every thread issues the tile's o loads of its
    // dimension d at once; meanwhile warp 0 loads the tile's (m_c, l_c), one
    // chunk per lane: the running maximum before chunk c is a prefix maximum
    // (exact in any order: a shuffle scan), and chunk c's merge factors
    // depend only on it and m_c, so each lane computes its chunk's factors.
    // Then each thread merges its o values in chunk order: the same
    // operations, in the same order, as a sequential walk over the chunks.
    constexpr int kTile = 32;
    __shared__ float fa[kTile];               // alpha of chunk c
    __shared__ float fb[kTile];               // beta of chunk c
    __shared__ float fl[kTile];               // l_c
    const int h = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int d = threadIdx.x;
    const float *w = p.ws + (b * p.Hq + h) * p.chunks * (kD + 2);
    // The first tile's loads go out before the sequence length is known: the
    // workspace holds p.chunks records a head, and records past the
    // sequence's chunks are loaded but never used.
    const int nt0 = min(kTile, p.chunks);
    float ov0[kTile];
#pragma unroll
    for (int c = 0; c < kTile; ++c) ov0[c] = c < nt0 ? w[static_cast<int64_t>(c) * (kD + 2) + 2 + d] : 0.0f;
    const float mc0 = d < nt0 ? w[static_cast<int64_t>(d) * (kD + 2)] : -INFINITY;
    const float lc0 = d < nt0 ? w[static_cast<int64_t>(d) * (kD + 2) + 1] : 0.0f;
    int L;
    if (!seq_ok(p, b, L)) return;
    const int nc = (L + kChunk - 1) / kChunk;
    if (!BI_IN_BOUNDS(nc <= p.chunks, p.status)) return;   // debug build: inside the workspace
    float o = 0.0f, l = 0.0f, m_run = -INFINITY;           // m_run: warp 0's copy of the running maximum
    // merge chunks c0 .. c0 + nt - 1 (their o values in ov; (m_c, l_c) of
    // chunk c0 + d in warp 0's lane d)
    auto merge_tile = [&](const float (&ov)[kTile], int nt, float mc, float lc) {
        __syncthreads();                                   // previous tile fully consumed
        if (d < 32) {
            mc = d < nt ? mc : -INFINITY;
            lc = d < nt ? lc : 0.0f;
            float incl = mc;                               // max(m_c0 .. m_c) over the tile
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, incl, off);
                if (d >= off) incl = fmaxf(incl, v);
            }
            float before = __shfl_up_sync(0xffffffffu, incl, 1);
            before = d == 0 ? m_run : fmaxf(m_run, before);   // running maximum before chunk c0 + d
            float mn, a, bt;
            merge_factors(before, mc, mn, a, bt);
            if (d < nt) {
                fa[d] = a;
                fb[d] = bt;
                fl[d] = lc;
            }
            m_run = fmaxf(m_run, __shfl_sync(0xffffffffu, incl, 31));
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
            if (c < nt) {
                o = merge_value(o, ov[c], fa[c], fb[c]);
                l = merge_value(l, fl[c], fa[c], fb[c]);
            }
        }
    };
    merge_tile(ov0, min(kTile, nc), mc0, lc0);
    for (int c0 = kTile; c0 < nc; c0 += kTile) {
        const int nt = min(kTile, nc - c0);
        const float *oc = w + static_cast<int64_t>(c0) * (kD + 2) + 2 + d;
        float ov[kTile];                                   // in flight while warp 0 prepares the factors
#pragma unroll
        for (int c = 0; c < kTile; ++c) ov[c] = c < nt ? oc[static_cast<int64_t>(c) * (kD + 2)] : 0.0f;
        const float *wc = w + static_cast<int64_t>(c0 + d) * (kD + 2);
        const float mc = d < nt ? wc[0] : -INFINITY;       // read by warp 0 only
        const float lc = d < nt ? wc[1] : 0.0f;
        merge_tile(ov, nt, mc, lc);
    }
    const float r = __fdiv_rn(o, l);
    const uint32_t packed = pack_bf16x2(__float_as_uint(r), 0u);
    p.O[(b * p.Hq + h) * kD + d] = static_cast<uint16_t>(packed & 0xFFFFu);
}

// ------------------------------------------------------------------ extend

constexpr int kExtRows = 128;                  // query rows (token, head) per CTA: one m16 tile per warp
constexpr int kExtThreads = 256;
// K and V tiles twice (the next chunk loads while this one is used), q rows,
// the K/V row offsets of three chunks.
constexpr int kExtSmem = 4 * kTileBytes + kExtRows * kD * 2 + 3 * kChunk * 8;

struct ExtParams {
    const uint16_t *Q;       // [total_q][Hq][D]
    const int32_t *cu_q;     // [B+1]
    const uint16_t *K;       // [blocks][bs][Hkv][D]
    const uint16_t *V;
    const int32_t *table;    // [B][max_blocks]
    const int32_t *lens;     // [B], cached length including the new tokens
    uint16_t *O;             // [total_q][Hq][D]
    int64_t num_blocks, batch;
    int32_t total_q, max_blocks, Hq, Hkv, bs, max_len, max_q;
    float scale;
    unsigned *status;
};

// Tensor-pipe turns of the extend kernel's two warp groups (named barriers
// 1 and 2, 256 threads: one group arrives, the other waits).
__device__ __forceinline__ void turn_wait(int id) { asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void turn_pass(int id) { asm volatile("bar.arrive %0, 256;" ::"r"(id) : "memory"); }

template <int G>
__global__ void __launch_bounds__(kExtThreads, 1)
attn_extend_kernel(const ExtParams p) {
    constexpr int kTQ = kExtRows / G;                  // query tokens per CTA
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *KV = smem;                                                    // [2][K, V] tiles, swizzled rows
    uint16_t *qb = reinterpret_cast<uint16_t *>(smem + 4 * kTileBytes);   // [kExtRows][kD] bf16
    int64_t *rowoff = reinterpret_cast<int64_t *>(qb + kExtRows * kD);     // [3][kChunk], -1: no row
    // blockIdx.x = (tile from the last, sequence, KV head): the tiles with the
    // latest tokens (the most chunks) of every sequence start first, so the
    // light ones fill the tail
    const int64_t per_tile = static_cast<int64_t>(p.batch) * p.Hkv;
    const int g = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.Hkv));
    const int64_t b = (blockIdx.x / static_cast<unsigned>(p.Hkv)) % p.batch;
    const int tile = static_cast<int>(gridDim.x / per_tile - 1 - blockIdx.x / per_tile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int L = p.lens[b];
    const int64_t qlen = q1 - q0;
    if (q0 < 0 || q1 < q0 || q1 > p.total_q || qlen > p.max_q || L < qlen || L > p.max_len ||
        L > static_cast<int64_t>(p.max_blocks) * p.bs) {
        if (tid == 0 && tile == 0 && g == 0) atomicOr(p.status, kDevBadOffsets);
        return;
    }
    const int i0 = tile * kTQ;                         // first query token of this CTA
    if (i0 >= qlen) return;
    const int ntok = static_cast<int>(qlen - i0 < kTQ ? qlen - i0 : static_cast<int64_t>(kTQ));
    const int base = L - static_cast<int>(qlen);       // position of query token 0
    const int L_last = base + i0 + ntok;               // the last token's causal length
    const int nchunks = (L_last + kChunk - 1) / kChunk;

    // q rows: row r = token r / G, head g*G + r % G (zero rows past the
    // tokens); 16-byte piece x of row r at piece x ^ (r % 8). Copied by
    // cp.async in chunk 0's group, so they travel while the block table is read.
    for (int i = tid; i < kExtRows * kD / 8; i += kExtThreads) {
        const int r = i / (kD / 8), x = i % (kD / 8);
        const bool v = r / G < ntok;
        cp_async_16(smem_u32(qb + r * kD + ((x ^ (r & 7)) * 8)),
                    v ? p.Q + ((q0 + i0 + r / G) * p.Hq + g * G + r % G) * kD + x * 8 : p.Q, v ? 16u : 0u);
    }
    // row offsets of chunk c's K/V rows (threads 0..127; buffer c % 3, so a
    // buffer is rewritten only after every warp has left the chunk that used it)
    auto chunk_rows = [&](int c) -> int {
        int bad = 0;
        if (tid < kChunk) {
            const int j = c * kChunk + tid;
            int64_t off = -1;
            if (j < L_last) {
                const int64_t blk = p.table[b * p.max_blocks + j / p.bs];
                if (blk >= 0 && blk < p.num_blocks) {
                    off = ((blk * p.bs + j % p.bs) * p.Hkv + g) * kD;
                } else {
                    atomicOr(p.status, kDevBadOffsets);
                    bad = 1;
                }
            }
            rowoff[(c % 3) * kChunk + tid] = off;
        }
        return bad;
    };
    auto issue_chunk = [&](int c) {                    // after chunk_rows(c) and a barrier
        const int buf = c & 1;
        const int64_t *ro = rowoff + (c % 3) * kChunk;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint16_t *src = which == 0 ? p.K : p.V;
            const uint32_t dst0 = smem_u32(KV + (2 * buf + which) * kTileBytes);
#pragma unroll
            for (int r = 0; r < kChunk * 16 / kExtThreads; ++r) {
                const int i = tid + r * kExtThreads;
                const int t = i >> 4, x = i & 15;
                const int64_t off = ro[t];
                cp_async_16(dst0 + t * kRowBytes + ((x ^ (t & 7)) << 4), off >= 0 ? src + off + x * 8 : src,
                            off >= 0 ? 16u : 0u);
            }
        }
        cp_async_commit();
    };
    // q rows and chunk 0's row offsets; bad_cur: chunk c has a token without a valid block
    int bad_cur = __syncthreads_or(chunk_rows(0));
    issue_chunk(0);

    const int gq = lane >> 2, cq = lane & 3;           // fragment row group, column pair
    const int rt = warp;                               // this warp's 16-row tile
    const int wg = warp >> 2;                          // warp group: 0 = A, 1 = B
    const int ra = rt * 16 + gq, rb = ra + 8;          // this thread's two rows
    // the warp's q fragments (A operand of q.k) come from shared memory by
    // ldmatrix: lane l addresses row (l / 8 % 2) * 8 + l % 8 of the tile,
    // 16-byte piece 2 ks + l / 16
    const int qrow = rt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
    const uint32_t qaddr = smem_u32(qb) + qrow * kRowBytes;
    // running state of rows ra (h = 0) and rb (h = 1), all 128 dimensions
    float o_run[kD / 8][4], m_run[2], l_run[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.0f;
    }
#pragma unroll
    for (int nt = 0; nt < kD / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_run[nt][e] = 0.0f;
    // the causal length of each row: position + 1 (0 for rows past the tokens)
    const int len_a = ra / G < ntok ? base + i0 + ra / G + 1 : 0;
    const int len_b = rb / G < ntok ? base + i0 + rb / G + 1 : 0;

    for (int c = 0; c < nchunks; ++c) {
        const int j0 = c * kChunk;
        const int64_t *ro = rowoff + (c % 3) * kChunk;
        const uint8_t *Ks = KV + (2 * (c & 1)) * kTileBytes;
        const uint8_t *Vs = KV + (2 * (c & 1) + 1) * kTileBytes;
        const bool more = c + 1 < nchunks;
        // every warp has left chunk c - 1 (its K/V buffer is free) and chunk
        // c + 1's row offsets are written
        const int bad_next = __syncthreads_or(more ? chunk_rows(c + 1) : 0);
        const bool bad = bad_cur != 0;
        bad_cur = bad_next;
        if (more) {
            issue_chunk(c + 1);
            cp_async_wait<1>();                        // this thread's copies of chunk c
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();                               // everyone's

        // tokens of this chunk each row sees (decode of the sequence cut after the row's token)
        const int na = max(0, min(kChunk, len_a - j0)), nb = max(0, min(kChunk, len_b - j0));
        // The two warp groups (warps 0-3, 4-7; warp w and w + 4 share a
        // scheduler) take turns on the tensor pipe: A's q.k, B's q.k, A's p.V,
        // B's p.V, ..., each group's softmax and merge running under the other
        // group's MMAs. Named barrier 1 hands the turn to A, 2 to B (bar.arrive
        // by the group that finishes a phase, bar.sync by the one that starts).
        // Every warp takes every turn and computes every chunk: rows that see
        // nothing of it score -inf, get p = 0 and skip the merge.
        if (wg == 1 || c > 0) turn_wait(wg == 0 ? 1 : 2);

        // scores s = scale * q . k for the tile's 16 rows and all 128 tokens,
        // dimensions
        // ascending in 16-dimension steps; tokens a row does not see are -inf.
        // s[nt][e]: row ra (e < 2) or rb, token 8 nt + 2 cq + (e & 1)
        // The 16 n-tiles' MMA chains are interleaved (dimension step outer),
        // each chain still in ascending dimension order.
        float s[kChunk / 8][4];
#pragma unroll
        for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] = 0.0f;
#pragma unroll
        for (int kp = 0; kp < kD / 32; ++kp) {                     // two 16-dimension steps per ldmatrix
            uint32_t qf[2][4];
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int piece = 2 * (2 * kp + k2) + (lane >> 4);
                ldmatrix_x4(qf[k2][0], qf[k2][1], qf[k2][2], qf[k2][3], qaddr + ((piece ^ (qrow & 7)) << 4));
            }
#pragma unroll
            for (int nt = 0; nt < kChunk / 8; ++nt) {
                const int trow = nt * 8 + (lane & 7);              // the K row this lane addresses
                const int chunk = 4 * kp + (lane >> 3);            // 16-byte chunk of matrix lane/8
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(b0, b1, b2, b3, smem_u32(Ks) + trow * kRowBytes + ((chunk ^ (trow & 7)) << 4));
                mma_16816(s[nt], qf[0][0], qf[0][1], qf[0][2], qf[0][3], b0, b1);
                mma_16816(s[nt], qf[1][0], qf[1][1], qf[1][2], qf[1][3], b2, b3);
            }
        }
        turn_pass(wg == 0 ? 2 : 1);
        // a chunk every row of the tile sees whole, with every block valid,
        // needs no masks
        const bool whole = !bad && __all_sync(0xffffffffu, na == kChunk && nb == kChunk);
        float m[2] = {-INFINITY, -INFINITY};
        if (whole) {
#pragma unroll
            for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[nt][e] = __fmul_rn(s[nt][e], p.scale);
                    m[e >> 1] = fmaxf(m[e >> 1], s[nt][e]);
                }
        } else {
#pragma unroll
            for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = nt * 8 + 2 * cq + (e & 1);
                    s[nt][e] = t < (e < 2 ? na : nb) ? (ro[t] >= 0 ? __fmul_rn(s[nt][e], p.scale) : -INFINITY)
                                                     : -INFINITY;
                    m[e >> 1] = fmaxf(m[e >> 1], s[nt][e]);
                }
        }
        // per row: max (any order gives the same value), then e^(s - m) for the
        // tokens it sees (0 past them)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            m[h] = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], 1));
            m[h] = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], 2));
        }
        if (whole) {
#pragma unroll
            for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = expf(s[nt][e] - m[e >> 1]);
        } else {
#pragma unroll
            for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = nt * 8 + 2 * cq + (e & 1);
                    s[nt][e] = t < (e < 2 ? na : nb) ? expf(s[nt][e] - m[e >> 1]) : 0.0f;
                }
        }
        // per row: the sum in decode's order. Lane L of decode sums tokens
        // L, L + 32, L + 64, L + 96 in turn, then a butterfly over lanes xor
        // 16, 8, 4, 2, 1. Here L = 8 (nt % 4) + 2 cq + (e & 1): the column
        // steps (nt + 4k) and the butterfly steps 16 and 8 (nt ^ 2, nt ^ 1) and
        // 1 (e ^ 1) are in this thread; steps 4 and 2 are lanes xor 2 and 1.
        // Each butterfly step adds two equal-rank partials, and a + b = b + a,
        // so every lane's total is the same bits as decode's.
        float l[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float x[2];
#pragma unroll
            for (int e0 = 0; e0 < 2; ++e0) {
                float col[4];
#pragma unroll
                for (int n4 = 0; n4 < 4; ++n4) {
                    float acc = s[n4][2 * h + e0];
#pragma unroll
                    for (int k = 1; k < 4; ++k) acc += s[n4 + 4 * k][2 * h + e0];
                    col[n4] = acc;
                }
                const float u0 = col[0] + col[2], u1 = col[1] + col[3];   // step 16
                float v = u0 + u1;                                        // step 8
                v += __shfl_xor_sync(0xffffffffu, v, 2);                  // step 4
                v += __shfl_xor_sync(0xffffffffu, v, 1);                  // step 2
                x[e0] = v;
            }
            l[h] = x[0] + x[1];                                           // step 1
        }

        turn_wait(wg == 0 ? 1 : 2);
        // values: O_c = sum_t p_t v_t for all 128 dimensions, p = hi + lo
        // (two bf16 MMAs per step), tokens ascending in 16-token steps; the
        // exponentials are already in the A-fragment layout
        float acc[kD / 8][4];
#pragma unroll
        for (int nt = 0; nt < kD / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        const int mi = lane >> 3, mr = lane & 7;       // ldmatrix: matrix, row
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t ph0, pl0, ph1, pl1, ph2, pl2, ph3, pl3;
            split_bf16x2(s[2 * ks][0], s[2 * ks][1], ph0, pl0);
            split_bf16x2(s[2 * ks][2], s[2 * ks][3], ph1, pl1);
            split_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1], ph2, pl2);
            split_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3], ph3, pl3);
            const int tok = ks * 16 + (mi & 1) * 8 + mr;
            // dimensions in two halves of 64 (four ldmatrix each); each
            // accumulator takes hi, then lo (the chains interleaved)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[4][4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {       // two 8-dimension tiles per ldmatrix
                    const int chunk = 2 * (4 * half + q4) + (mi >> 1);
                    ldmatrix_x4_trans(v[q4][0], v[q4][1], v[q4][2], v[q4][3],
                                      smem_u32(Vs + tok * kRowBytes + ((chunk ^ (tok & 7)) << 4)));
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int np = 4 * half + q4;
                    mma_16816(acc[2 * np], ph0, ph1, ph2, ph3, v[q4][0], v[q4][1]);
                    mma_16816(acc[2 * np + 1], ph0, ph1, ph2, ph3, v[q4][2], v[q4][3]);
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int np = 4 * half + q4;
                    mma_16816(acc[2 * np], pl0, pl1, pl2, pl3, v[q4][0], v[q4][1]);
                    mma_16816(acc[2 * np + 1], pl0, pl1, pl2, pl3, v[q4][2], v[q4][3]);
                }
            }
        }
        turn_pass(wg == 0 ? 2 : 1);
        // merge this chunk into the rows' running state, in chunk order
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if ((h ? nb : na) == 0) continue;
            float mn, al, be;
            merge_factors(m_run[h], m[h], mn, al, be);
            m_run[h] = mn;
            l_run[h] = merge_value(l_run[h], l[h], al, be);
#pragma unroll
            for (int nt = 0; nt < kD / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    o_run[nt][2 * h + e] = merge_value(o_run[nt][2 * h + e], acc[nt][2 * h + e], al, be);
        }
    }

    if (wg == 0) turn_wait(1);                            // B's hand-over after its last p.V

    // o / l, rounded to bf16, for the rows that exist
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h ? rb : ra;
        if (r / G >= ntok || !BI_IN_BOUNDS(q0 + i0 + r / G < p.total_q, p.status)) continue;
        uint16_t *orow = p.O + ((q0 + i0 + r / G) * p.Hq + g * G + r % G) * kD + 2 * cq;
#pragma unroll
        for (int nt = 0; nt < kD / 8; ++nt) {
            const float x0 = __fdiv_rn(o_run[nt][2 * h], l_run[h]);
            const float x1 = __fdiv_rn(o_run[nt][2 * h + 1], l_run[h]);
            *reinterpret_cast<uint32_t *>(orow + nt * 8) = pack_bf16x2(__float_as_uint(x0), __float_as_uint(x1));
        }
    }
}

}  // namespace

int64_t attention_decode_workspace_bytes(int64_t B, int32_t Hq, int32_t max_len) {
    if (B < 0 || Hq < 1 || max_len < 1) return -1;
    const int64_t chunks = (static_cast<int64_t>(max_len) + kChunk - 1) / kChunk;
    constexpr int64_t kRecord = (kD + 2) * static_cast<int64_t>(sizeof(float));   // (m, l, o) of one head and chunk
    // -1 when the size does not fit in an int64_t
    const int64_t records_max = INT64_MAX / kRecord;
    if (B > records_max / Hq || B * Hq > records_max / chunks) return -1;
    return B * Hq * chunks * kRecord;
}

template <int G, int SLOTS, int NG>
bi_status launch_split_shape(const dim3 &grid, const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p,
                             cudaStream_t s) {
    static unsigned long long configured = 0;
    constexpr int smem = dec_smem<SLOTS, NG>();
    if (ensure_smem_attr(reinterpret_cast<const void *>(attn_split_kernel<G, SLOTS, NG>), smem, &configured) != BI_OK)
        return BI_ERR_CUDA;
    return launch_pdl(attn_split_kernel<G, SLOTS, NG>, grid, dim3(dec_threads<SLOTS>()), smem, s, tmK, tmV, p);
}
// At most two items per SM: one item per CTA, two CTAs per SM; else the ring.
template <int G>
bi_status launch_split(int64_t items, int sms, const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnParams &p,
                       cudaStream_t s) {
    if (items <= 2 * static_cast<int64_t>(sms))
        return launch_split_shape<G, 1, 1>(dim3(static_cast<unsigned>(items)), tmK, tmV, p, s);
    return launch_split_shape<G, 3, 2>(dim3(static_cast<unsigned>(sms)), tmK, tmV, p, s);
}
#define SPLIT_LAUNCH(G)                                              \
    do {                                                             \
        const bi_status st_ = launch_split<G>(items, info->sm_count, tmK, tmV, p, s); \
        if (st_ != BI_OK) return st_;                                \
    } while (0)

bi_status launch_attention_decode(const void *Q, const void *K, const void *V, const int32_t *table,
                                  int32_t max_blocks, int64_t num_blocks, const int32_t *lens, int64_t B, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t bs, int32_t max_len, float scale, void *workspace,
                                  void *O, cudaStream_t s) {
    (void)D;
    AttnParams p{};
    p.Q = static_cast<const uint16_t *>(Q);
    p.K = static_cast<const uint16_t *>(K);
    p.V = static_cast<const uint16_t *>(V);
    p.table = table;
    p.lens = lens;
    p.ws = static_cast<float *>(workspace);
    p.O = static_cast<uint16_t *>(O);
    p.num_blocks = num_blocks;
    p.batch = B;
    p.max_blocks = max_blocks;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = bs;
    p.chunks = static_cast<int32_t>((static_cast<int64_t>(max_len) + kChunk - 1) / kChunk);
    p.max_len = max_len;
    p.scale = scale;
    p.status = device_status_word();
    const int G = Hq / Hkv;
    int dev = 0;
    const DeviceInfo *info = nullptr;
    if (current_device(&dev, &info) != BI_OK) return BI_ERR_CUDA;
    const int64_t items = B * Hkv * static_cast<int64_t>(p.chunks);
    // TMA boxes of whole cache blocks (box start rows on 1024-byte swizzle atoms)
    CUtensorMap tmK{}, tmV{};
    p.box_rows = bs % kChunk == 0 ? kChunk : (kChunk % bs == 0 && bs >= 8 ? bs : 0);
    if (p.box_rows > 0) {
        const uint64_t dims[4] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(bs),
                                  static_cast<uint64_t>(num_blocks)};
        const uint64_t strides[3] = {static_cast<uint64_t>(kRowBytes), static_cast<uint64_t>(Hkv) * kRowBytes,
                                     static_cast<uint64_t>(bs) * Hkv * kRowBytes};
        const uint32_t box[4] = {64, 1, static_cast<uint32_t>(p.box_rows), 1};
        if (make_tmap_4d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) != BI_OK ||
            make_tmap_4d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) != BI_OK)
            p.box_rows = 0;                          // the per-row copies need no tensor map
    }
    switch (G) {
        case 1: SPLIT_LAUNCH(1); break;
        case 2: SPLIT_LAUNCH(2); break;
        case 4: SPLIT_LAUNCH(4); break;
        case 8: SPLIT_LAUNCH(8); break;
        default: return BI_ERR_UNSUPPORTED;
    }
    return launch_pdl(attn_combine_kernel, dim3(Hq, static_cast<unsigned>(B)), dim3(kCombineThreads), 0, s, p);
}

template <int G>
bi_status launch_extend_g(const dim3 &grid, const ExtParams &p, cudaStream_t s) {
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(attn_extend_kernel<G>), kExtSmem, &configured) != BI_OK)
        return BI_ERR_CUDA;
    return launch_pdl(attn_extend_kernel<G>, grid, dim3(kExtThreads), kExtSmem, s, p);
}

bi_status launch_attention_extend(const void *Q, const int32_t *cu_q, int32_t total_q, const void *K, const void *V,
                                  const int32_t *table, int32_t max_blocks, int64_t num_blocks, const int32_t *lens,
                                  int64_t B, int32_t Hq, int32_t Hkv, int32_t bs, int32_t max_len, int32_t max_q,
                                  float scale, void *O, cudaStream_t s) {
    ExtParams p{};
    p.Q = static_cast<const uint16_t *>(Q);
    p.cu_q = cu_q;
    p.K = static_cast<const uint16_t *>(K);
    p.V = static_cast<const uint16_t *>(V);
    p.table = table;
    p.lens = lens;
    p.O = static_cast<uint16_t *>(O);
    p.num_blocks = num_blocks;
    p.batch = B;
    p.total_q = total_q;
    p.max_blocks = max_blocks;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = bs;
    p.max_len = max_len;
    p.max_q = max_q;
    p.scale = scale;
    p.status = device_status_word();
    const int G = Hq / Hkv;
    const int tq = kExtRows / G;
    const int64_t ctas_x = (static_cast<int64_t>(max_q) + tq - 1) / tq * B * Hkv;   // (tile, sequence, KV head)
    if (ctas_x > 0x7fffffff) return BI_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(ctas_x));
    switch (G) {
        case 1: return launch_extend_g<1>(grid, p, s);
        case 2: return launch_extend_g<2>(grid, p, s);
        case 4: return launch_extend_g<4>(grid, p, s);
        case 8: return launch_extend_g<8>(grid, p, s);
        default: return BI_ERR_UNSUPPORTED;
    }
}

}  // namespace bi

// ---------------------------------------------------------------------------
// Allocation-free variant of bi_attention_decode.
//
// Some callers cannot call cudaMalloc: for example code linked into a host
// program whose allocator has already reserved all device memory up front, or
// code on a latency-critical path that must not risk the device-wide
// synchronisation an allocation can cause. bi_attention_decode_noalloc gives
// them the same decode attention without a workspace argument: the per-chunk
// partial results go to the fixed array below instead. The array lives in
// device memory for as long as the library is loaded, on every GPU that loads
// it, so its size is kept modest and larger problems are refused.
//
// Every call shares the one array, and nothing in it needs to start at zero:
// the split kernel writes every entry the combine kernel later reads. The
// array keeps whatever the last call left in it. Two calls whose kernels
// overlap on the GPU (for example on different streams) race on it.
// ---------------------------------------------------------------------------
namespace bi {
namespace {

constexpr size_t kNoAllocScratchBytes = BI_ATTENTION_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxScratchDevices = 64;
std::once_flag g_scratch_once[kMaxScratchDevices];
void *g_scratch_ptr[kMaxScratchDevices];
cudaError_t g_scratch_err[kMaxScratchDevices];

// Device address of the array for the current device, looked up once per
// device (with that device current) on the first call made on it.
bi_status noalloc_scratch(void **ptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return BI_ERR_CUDA;
    std::call_once(g_scratch_once[dev], [dev] {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_scratch_ptr[dev] = p;
    });
    if (g_scratch_err[dev] != cudaSuccess || !g_scratch_ptr[dev]) return BI_ERR_CUDA;
    *ptr = g_scratch_ptr[dev];
    return BI_OK;
}

}  // namespace
}  // namespace bi

extern "C" bi_status bi_attention_decode_noalloc(const void *Q, const void *K_cache, const void *V_cache,
                                                 const int32_t *block_table, int32_t max_blocks_per_seq,
                                                 int64_t num_blocks, const int32_t *seq_lens, int64_t B, int32_t Hq,
                                                 int32_t Hkv, int32_t head_dim, int32_t block_size,
                                                 int32_t max_seq_len, float scale, void *O, bi_stream stream) {
    using namespace bi;
    if (B < 0 || B > 65535 || Hq < 1 || Hkv < 1 || block_size < 1 || max_seq_len < 1 ||
        max_seq_len > BI_ATTENTION_MAX_SEQ_LEN || max_blocks_per_seq < 1 || num_blocks < 1 || !(scale == scale))
        return BI_ERR_INVALID_ARG;
    if (B == 0) return BI_OK;
    if (!Q || !K_cache || !V_cache || !block_table || !seq_lens || !O) return BI_ERR_INVALID_ARG;
    if (head_dim != 128 || Hq % Hkv != 0) return BI_ERR_UNSUPPORTED;
    const int32_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return BI_ERR_UNSUPPORTED;
    // the problem's partial results must fit in the fixed array
    const int64_t need = attention_decode_workspace_bytes(B, Hq, max_seq_len);
    if (need < 0 || need > static_cast<int64_t>(kNoAllocScratchBytes)) return BI_ERR_UNSUPPORTED;
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const auto a4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(Q) || !a16(K_cache) || !a16(V_cache) || !a16(O) || !a4(block_table) || !a4(seq_lens))
        return BI_ERR_MISALIGNED;
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != BI_OK) return st;
    return launch_attention_decode(Q, K_cache, V_cache, block_table, max_blocks_per_seq, num_blocks, seq_lens, B, Hq,
                                   Hkv, head_dim, block_size, max_seq_len, scale, scratch, O,
                                   static_cast<cudaStream_t>(stream));
}
