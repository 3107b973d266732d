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
// Step 1, one CTA per (sequence, KV head, chunk), 128 threads, head_dim 128,
//   the G = Hq/Hkv query heads of the KV head together (GQA):
//   - scores: warp w takes tokens w, w+4, ...; lane l holds dims 4l..4l+3;
//     per head, the 4 products are added in order and the 32 lane sums by a
//     fixed xor butterfly; s = scale * q.k;
//   - per head (one warp each): m = max s (exact), p = exp(s - m), l = sum p
//     (lane-sequential, then butterfly);
//   - values: thread t owns dimension t and adds p_j v_j[t] over the chunk's
//     tokens in increasing order, for every head;
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
constexpr int kChunk = 256;
constexpr int kThreads = 128;
constexpr int kMaxGroup = 8;

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
    __shared__ float qs[G][kD];
    __shared__ float S[G][kChunk];
    __shared__ float ml[G][2];
    const int c = blockIdx.x, g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L;
    if (!seq_ok(p, b, L)) {
        if (threadIdx.x == 0 && c == 0 && g == 0) atomicOr(p.status, kDevBadOffsets);
        return;
    }
    const int j0 = c * kChunk;
    if (j0 >= L) return;                                  // this sequence has fewer chunks
    const int n = min(kChunk, L - j0);

    for (int i = threadIdx.x; i < G * kD; i += kThreads) {
        const int h = i / kD, d = i % kD;
        qs[h][d] = bf_at(p.Q + (b * p.Hq + g * G + h) * kD, d);
    }
    __syncthreads();

    // scores
    bool bad = false;
    for (int t = warp; t < n; t += kThreads / 32) {
        const int j = j0 + t;
        const int64_t blk = p.table[b * p.max_blocks + j / p.bs];
        if (blk < 0 || blk >= p.num_blocks) {
            bad = true;
            if (lane == 0)
                for (int h = 0; h < G; ++h) S[h][t] = -INFINITY;
            continue;
        }
        const uint16_t *k = p.K + ((blk * p.bs + j % p.bs) * p.Hkv + g) * kD;
        const uint2 kv = *reinterpret_cast<const uint2 *>(k + 4 * lane);
        const float k0 = bf_lo(kv.x), k1 = bf_hi(kv.x), k2 = bf_lo(kv.y), k3 = bf_hi(kv.y);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = qs[h][4 * lane] * k0;
            s = __fmaf_rn(qs[h][4 * lane + 1], k1, s);
            s = __fmaf_rn(qs[h][4 * lane + 2], k2, s);
            s = __fmaf_rn(qs[h][4 * lane + 3], k3, s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) S[h][t] = __fmul_rn(s, p.scale);
        }
    }
    if (bad && lane == 0) atomicOr(p.status, kDevBadOffsets);
    __syncthreads();

    // per head: max, exponentials, sum (head h on warp h % 4)
    for (int h = warp; h < G; h += kThreads / 32) {
        float m = -INFINITY;
        for (int t = lane; t < n; t += 32) m = fmaxf(m, S[h][t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.0f;
        for (int t = lane; t < n; t += 32) {
            const float e = expf(S[h][t] - m);
            S[h][t] = e;
            l += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            ml[h][0] = m;
            ml[h][1] = l;
        }
    }
    __syncthreads();

    // values: thread t owns dimension t
    const int d = threadIdx.x;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    for (int t = 0; t < n; ++t) {
        const int j = j0 + t;
        const int64_t blk = p.table[b * p.max_blocks + j / p.bs];
        if (blk < 0 || blk >= p.num_blocks) continue;
        const float v = bf_at(p.V + ((blk * p.bs + j % p.bs) * p.Hkv + g) * kD, d);
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = __fmaf_rn(S[h][t], v, acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float *w = p.ws + (((b * p.Hq + g * G + h) * p.chunks) + c) * (kD + 2);
        w[2 + d] = acc[h];
        if (d == 0) {
            w[0] = ml[h][0];
            w[1] = ml[h][1];
        }
    }
}

__global__ void __launch_bounds__(kThreads)
attn_combine_kernel(const AttnParams p) {
    const int h = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int d = threadIdx.x;
    int L;
    if (!seq_ok(p, b, L)) return;
    const int nc = (L + kChunk - 1) / kChunk;
    const float *w = p.ws + (b * p.Hq + h) * p.chunks * (kD + 2);
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, w[c * (kD + 2)]);
    float num = 0.0f, den = 0.0f;
    for (int c = 0; c < nc; ++c) {
        const float f = expf(w[c * (kD + 2)] - M);
        num = __fmaf_rn(f, w[c * (kD + 2) + 2 + d], num);
        den = __fmaf_rn(f, w[c * (kD + 2) + 1], den);
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
        case 1: attn_split_kernel<1><<<grid1, kThreads, 0, s>>>(p); break;
        case 2: attn_split_kernel<2><<<grid1, kThreads, 0, s>>>(p); break;
        case 4: attn_split_kernel<4><<<grid1, kThreads, 0, s>>>(p); break;
        case 8: attn_split_kernel<8><<<grid1, kThreads, 0, s>>>(p); break;
        default: return BI_ERR_UNSUPPORTED;
    }
    attn_combine_kernel<<<dim3(Hq, static_cast<unsigned>(B)), kThreads, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? BI_OK : BI_ERR_CUDA;
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
