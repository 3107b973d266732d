// attention.cu -- batch-invariant decode attention over a paged KV cache.
//
// Batch-invariant attention is on the vLLM tracking issue's TODO list
// (FlashInfer, TRITON_MLA, FLASHINFER_MLA support) and the vllm-ascend guide
// lists batch-invariant attention operators. Split-KV ("flash decoding")
// kernels usually pick the number of KV splits from the batch size to fill the
// GPU; that makes a sequence's reduction order depend on the batch. Here the
// split is fixed: a sequence's KV is cut into chunks of kChunk = 256 tokens by
// position alone, every chunk is reduced by one CTA in a fixed order, and the
// chunk results are merged in chunk order. Nothing a sequence sees depends on
// the other sequences in the batch.
//
// Step 1, one CTA per (sequence, KV head, chunk of kChunk = 128 tokens),
//   256 threads, head_dim 128, the G = Hq/Hkv query heads of the KV head
//   together (GQA):
//   - every thread issues its share of the chunk's K rows, then V rows, as
//     16-byte cp.async copies into shared memory (32 KB each; rows past the
//     sequence or in an invalid block are zero-filled), so the whole chunk is
//     in flight at once and three CTAs share an SM;
//   - scores, once K has landed: one lane per token, the 128 bf16 products
//     q[d] k[d] added in dimension order by fp32 FMAs on the bf16 operands
//     (each warp group of 4 takes every other head); s = scale * q.k;
//   - per head (warp h): m = max s (exact), p = exp(s - m), l = sum p
//     (lane-strided, then butterfly);
//   - values, once V has landed: thread (pair of dims, head group) adds
//     p_t v_t over the chunk's tokens in increasing order;
//   - writes fp32 (m, l, o[0..127]) per head and chunk to the workspace.
// Step 2, one CTA per (sequence, query head): M = max_c m_c; the output is
//   sum_c e^{m_c - M} o_c / sum_c e^{m_c - M} l_c, chunks in order, rounded to bf16.
#include <cuda_bf16.h>

#include <mutex>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 128;                    // tokens per chunk: fixed, by position
constexpr int kThreads = 256;                  // split kernel
constexpr int kWarps = kThreads / 32;
constexpr int kCombineThreads = 128;           // one thread per output dimension
constexpr int kRowBytes = kD * 2;              // one token's K (or V) row of one KV head
constexpr int kTileBytes = kChunk * kRowBytes; // 32 KB

// K and V tiles, then q (G x kD fp32), scores (G x kChunk fp32), (m, l) per
// head and the K-row offset of every token of the chunk. The value phase's
// partial sums (kThreads x G x 8 fp32) reuse the K and V tiles.
template <int G>
constexpr int split_smem_bytes() {
    return 2 * kTileBytes + (G * kD + G * kChunk + 2 * G) * 4 + kChunk * 8;
}
static_assert(kThreads * 8 * 8 * 4 <= 2 * kTileBytes, "value partials must fit in the K and V tiles");

// acc + a.lo * b.lo, then + a.hi * b.hi, each one fp32 FMA on bf16 operands
// (the product of two bf16 values is exact in fp32, so this is the same as
// widening both to fp32 first).
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(b));
    return acc;
}

// 16-byte global -> shared copy; src_bytes = 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf_at(const uint16_t *p, int i) { return __uint_as_float(static_cast<uint32_t>(p[i]) << 16); }

struct AttnParams {
    const uint16_t *Q;       // [B][Hq][D]
    const uint16_t *K;       // [blocks][bs][Hkv][D]
    const uint16_t *V;
    const int32_t *table;    // [B][max_blocks]
    const int32_t *lens;     // [B]
    float *ws;               // [B][Hq][chunks][kD + 2]
    uint16_t *O;             // [B][Hq][D]
    int64_t num_blocks;
    int32_t max_blocks, Hq, Hkv, bs, chunks, max_len;
    float scale;
    unsigned *status;
};

__device__ __forceinline__ bool seq_ok(const AttnParams &p, int64_t b, int &L) {
    L = p.lens[b];
    return L >= 1 && L <= p.max_len && L <= static_cast<int64_t>(p.max_blocks) * p.bs;
}

template <int G>
__global__ void __launch_bounds__(kThreads)
attn_split_kernel(const AttnParams p) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *Ks = smem;                                            // [kChunk][kD] bf16, 16-byte chunks swizzled
    uint8_t *Vs = smem + kTileBytes;                               // [kChunk][kD] bf16
    float *qs = reinterpret_cast<float *>(smem + 2 * kTileBytes);  // [G][kD] bf16 (first half used)
    uint16_t *qb = reinterpret_cast<uint16_t *>(qs);
    float *S = qs + G * kD;                                        // [kChunk][G]
    float *ml = S + G * kChunk;                                    // [G][2]
    int64_t *rowoff = reinterpret_cast<int64_t *>(ml + 2 * G);     // [kChunk], -1: no row
    float *part = reinterpret_cast<float *>(smem);                 // value partials, after the tiles are read
    const int c = blockIdx.x, g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int L;
    if (!seq_ok(p, b, L)) {
        if (tid == 0 && c == 0 && g == 0) atomicOr(p.status, kDevBadOffsets);
        return;
    }
    const int j0 = c * kChunk;
    if (j0 >= L) return;                                  // this sequence has fewer chunks
    const int n = min(kChunk, L - j0);

    // element offset of each token's K (and V) row for KV head g
    if (tid < kChunk) {
        int64_t off = -1;
        if (tid < n) {
            const int j = j0 + tid;
            const int64_t blk = p.table[b * p.max_blocks + j / p.bs];
            if (blk >= 0 && blk < p.num_blocks)
                off = ((blk * p.bs + j % p.bs) * p.Hkv + g) * kD;
            else
                atomicOr(p.status, kDevBadOffsets);
        }
        rowoff[tid] = off;
    }
    for (int i = tid; i < G * kD; i += kThreads) qb[i] = p.Q[(b * p.Hq + g * G) * kD + i];
    __syncthreads();

    // K rows (chunk x of row t at chunk x ^ (t % 8)), then V rows; missing rows are zero-filled
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const uint16_t *base = which == 0 ? p.K : p.V;
        const uint32_t dst0 = smem_u32(which == 0 ? Ks : Vs);
#pragma unroll
        for (int r = 0; r < kChunk * 16 / kThreads; ++r) {
            const int i = tid + r * kThreads;
            const int t = i >> 4, x = i & 15;
            const int64_t off = rowoff[t];
            const int xs = which == 0 ? (x ^ (t & 7)) : x;
            cp_async_16(dst0 + t * kRowBytes + xs * 16, off >= 0 ? base + off + x * 8 : base, off >= 0 ? 16u : 0u);
        }
        cp_async_commit();
    }
    cp_async_wait<1>();                                   // this thread's K copies
    __syncthreads();                                      // everyone's

    // scores: lane = token (t = 32*(warp%4) + lane), warp/4 picks every other head;
    // q.k adds the 128 products in dimension order
    {
        const int t = (warp & 3) * 32 + lane;
        const int h0 = warp >> 2;
        if (G > 1 || h0 == 0) {
            constexpr int NH = G > 1 ? G / 2 : 1;
            float acc[NH];
#pragma unroll
            for (int i = 0; i < NH; ++i) acc[i] = 0.0f;
            const uint8_t *krow = Ks + t * kRowBytes;
#pragma unroll 4
            for (int x = 0; x < 16; ++x) {
                const uint4 kv = *reinterpret_cast<const uint4 *>(krow + ((x ^ (t & 7)) << 4));
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    const uint4 qv = *reinterpret_cast<const uint4 *>(qb + (h0 + (G > 1 ? 2 * i : 0)) * kD + x * 8);
                    float sc = acc[i];
                    sc = fma_bf16x2(qv.x, kv.x, sc);
                    sc = fma_bf16x2(qv.y, kv.y, sc);
                    sc = fma_bf16x2(qv.z, kv.z, sc);
                    sc = fma_bf16x2(qv.w, kv.w, sc);
                    acc[i] = sc;
                }
            }
            if (t < n) {
                const bool valid = rowoff[t] >= 0;
#pragma unroll
                for (int i = 0; i < NH; ++i)
                    S[t * G + h0 + (G > 1 ? 2 * i : 0)] = valid ? __fmul_rn(acc[i], p.scale) : -INFINITY;
            }
        }
    }
    __syncthreads();

    // per head: max, exponentials, sum (head h on warp h)
    if (warp < G) {
        const int h = warp;
        float m = -INFINITY;
        for (int t = lane; t < n; t += 32) m = fmaxf(m, S[t * G + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
        for (int t = lane; t < n; t += 32) {
            const float e = expf(S[t * G + h] - m);
            S[t * G + h] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            ml[2 * h] = m;
            ml[2 * h + 1] = l;
        }
    }
    cp_async_wait<0>();                                   // this thread's V copies
    __syncthreads();

    // values: thread (dims 8*dg .. 8*dg+7, token group tg) adds p_t v_t over
    // tokens tg, tg+16, ... in order, for every head; the 16 token groups'
    // partial sums are then added in group order
    const int dg = tid & 15, tg = tid >> 4;
    float acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[h][k] = 0.0f;
#pragma unroll 2
    for (int t = tg; t < n; t += 16) {
        const uint4 vv = *reinterpret_cast<const uint4 *>(Vs + t * kRowBytes + dg * 16);
        const float v[8] = {bf_lo(vv.x), bf_hi(vv.x), bf_lo(vv.y), bf_hi(vv.y),
                            bf_lo(vv.z), bf_hi(vv.z), bf_lo(vv.w), bf_hi(vv.w)};
        float e[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
            for (int h = 0; h < G; h += 4) {
                const float4 e4 = *reinterpret_cast<const float4 *>(S + t * G + h);
                e[h] = e4.x, e[h + 1] = e4.y, e[h + 2] = e4.z, e[h + 3] = e4.w;
            }
        } else {
#pragma unroll
            for (int h = 0; h < G; ++h) e[h] = S[t * G + h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[h][k] = __fmaf_rn(e[h], v[k], acc[h][k]);
    }
    __syncthreads();                                      // tiles no longer read: reuse them
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float4 *dst = reinterpret_cast<float4 *>(part + (tg * G + h) * kD + dg * 8);
        dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
    __syncthreads();
    for (int o = tid; o < G * kD; o += kThreads) {
        const int h = o / kD, d = o % kD;
        float sum = part[h * kD + d];
#pragma unroll
        for (int gg = 1; gg < 16; ++gg) sum += part[(gg * G + h) * kD + d];
        float *w = p.ws + (((b * p.Hq + g * G + h) * p.chunks) + c) * (kD + 2);
        w[2 + d] = sum;
        if (d == 0) {
            w[0] = ml[2 * h];
            w[1] = ml[2 * h + 1];
        }
    }
}

__global__ void __launch_bounds__(kCombineThreads)
attn_combine_kernel(const AttnParams p) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    // Chunk statistics go through shared memory in tiles of kCombineThreads
    // chunks, loaded in parallel; the arithmetic is the sequential chunk-order
    // merge described at the top of the file (the maximum is exact in any order).
    __shared__ float red[kCombineThreads / 32];
    __shared__ float fw[kCombineThreads];     // e^{m_c - M} for the tile's chunks
    __shared__ float fl[kCombineThreads];     // l_c
    const int h = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
    int L;
    if (!seq_ok(p, b, L)) return;
    const int nc = (L + kChunk - 1) / kChunk;
    const float *w = p.ws + (b * p.Hq + h) * p.chunks * (kD + 2);
    float m = -INFINITY;
    for (int c = d; c < nc; c += kCombineThreads) m = fmaxf(m, w[static_cast<int64_t>(c) * (kD + 2)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int i = 1; i < kCombineThreads / 32; ++i) M = fmaxf(M, red[i]);
    float num = 0.0f, den = 0.0f;
    for (int c0 = 0; c0 < nc; c0 += kCombineThreads) {
        const int nt = min(kCombineThreads, nc - c0);
        __syncthreads();                                   // previous tile fully consumed
        if (d < nt) {
            const float *wc = w + static_cast<int64_t>(c0 + d) * (kD + 2);
            fw[d] = expf(wc[0] - M);
            fl[d] = wc[1];
        }
        __syncthreads();
        const float *oc = w + static_cast<int64_t>(c0) * (kD + 2) + 2 + d;
        int c = 0;
        for (; c + 8 <= nt; c += 8) {                      // 8 independent loads in flight
            float o8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o8[i] = oc[static_cast<int64_t>(c + i) * (kD + 2)];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                num = __fmaf_rn(fw[c + i], o8[i], num);
                den = __fmaf_rn(fw[c + i], fl[c + i], den);
            }
        }
        for (; c < nt; ++c) {
            num = __fmaf_rn(fw[c], oc[static_cast<int64_t>(c) * (kD + 2)], num);
            den = __fmaf_rn(fw[c], fl[c], den);
        }
    }
    const float o = __fdiv_rn(num, den);
    const uint32_t packed = pack_bf16x2(__float_as_uint(o), 0u);
    p.O[(b * p.Hq + h) * kD + d] = static_cast<uint16_t>(packed & 0xFFFFu);
}

}  // namespace

int64_t attention_decode_workspace_bytes(int64_t B, int32_t Hq, int32_t max_len) {
    const int64_t chunks = (max_len + kChunk - 1) / kChunk;
    return B * Hq * chunks * (kD + 2) * static_cast<int64_t>(sizeof(float));
}

template <int G>
bi_status launch_split(const dim3 &grid, const AttnParams &p, cudaStream_t s) {
    static unsigned long long configured = 0;
    if (ensure_smem_attr(reinterpret_cast<const void *>(attn_split_kernel<G>), split_smem_bytes<G>(), &configured) !=
        BI_OK)
        return BI_ERR_CUDA;
    return launch_pdl(attn_split_kernel<G>, grid, dim3(kThreads), split_smem_bytes<G>(), s, p);
}
#define SPLIT_LAUNCH(G)                                    \
    do {                                                   \
        const bi_status st_ = launch_split<G>(grid1, p, s); \
        if (st_ != BI_OK) return st_;                      \
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
    p.max_blocks = max_blocks;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = bs;
    p.chunks = (max_len + kChunk - 1) / kChunk;
    p.max_len = max_len;
    p.scale = scale;
    p.status = device_status_word();
    const int G = Hq / Hkv;
    const dim3 grid1(p.chunks, Hkv, static_cast<unsigned>(B));
    switch (G) {
        case 1: SPLIT_LAUNCH(1); break;
        case 2: SPLIT_LAUNCH(2); break;
        case 4: SPLIT_LAUNCH(4); break;
        case 8: SPLIT_LAUNCH(8); break;
        default: return BI_ERR_UNSUPPORTED;
    }
    return launch_pdl(attn_combine_kernel, dim3(Hq, static_cast<unsigned>(B)), dim3(kCombineThreads), 0, s, p);
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
    if (B < 0 || B > 65535 || Hq < 1 || Hkv < 1 || block_size < 1 || max_seq_len < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || !(scale == scale))
        return BI_ERR_INVALID_ARG;
    if (B == 0) return BI_OK;
    if (!Q || !K_cache || !V_cache || !block_table || !seq_lens || !O) return BI_ERR_INVALID_ARG;
    if (head_dim != 128 || Hq % Hkv != 0) return BI_ERR_UNSUPPORTED;
    const int32_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return BI_ERR_UNSUPPORTED;
    // the problem's partial results must fit in the fixed array
    if (attention_decode_workspace_bytes(B, Hq, max_seq_len) > static_cast<int64_t>(kNoAllocScratchBytes))
        return BI_ERR_UNSUPPORTED;
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
