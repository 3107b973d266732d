// abi.cu -- the C ABI of libbi: argument checks, device facts, the device
// status word, tensor-map encoding and the extern "C" entry points.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <functional>
#include <mutex>

#include "bi_internal.h"

namespace bi {
namespace {


// One status word per device; kernels or codes into it, bi_device_status
// reads and clears it.
__device__ unsigned g_status_word;

struct DeviceSlot {
    std::once_flag once;
    DeviceInfo info;
    bi_status init_status = BI_ERR_CUDA;
    unsigned *status = nullptr;
};
DeviceSlot g_devices[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void init_device(int dev, DeviceSlot &slot) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&slot.info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&slot.info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        slot.init_status = BI_ERR_CUDA;
        return;
    }
    slot.info.is_sm103 = (major == 10 && minor == 3);
    if (!slot.info.is_sm103) {
        slot.init_status = BI_ERR_ARCH;
        return;
    }
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
        slot.init_status = BI_ERR_CUDA;
        return;
    }
    slot.status = static_cast<unsigned *>(addr);
    slot.init_status = BI_OK;
}

}  // namespace

bi_status current_device(int *dev, const DeviceInfo **info) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return BI_ERR_CUDA;
    DeviceSlot &slot = g_devices[*dev];
    std::call_once(slot.once, init_device, *dev, std::ref(slot));
    *info = &slot.info;
    return slot.init_status;
}

unsigned *device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    return g_devices[dev].status;
}

bi_status ensure_smem_attr(const void *kernel, int bytes, unsigned long long *done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BI_ERR_CUDA;
    const unsigned long long bit = 1ull << dev;
    auto *flag = reinterpret_cast<std::atomic<unsigned long long> *>(done);
    if (flag->load(std::memory_order_acquire) & bit) return BI_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return BI_ERR_CUDA;
    flag->fetch_or(bit, std::memory_order_acq_rel);
    return BI_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bi_status make_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                       uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                       CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return BI_ERR_CUDA;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

bi_status make_tmap_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t dims[3],
                       const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return BI_ERR_CUDA;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t s[2] = {strides_bytes[0], strides_bytes[1]};
    const cuuint32_t b[3] = {box[0], box[1], box[2]};
    const cuuint32_t e[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

bi_status make_tmap_4d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc) return BI_ERR_CUDA;
    const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    const cuuint64_t s[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
    const cuuint32_t e[4] = {1, 1, 1, 1};
    CUresult r = enc(map, dtype, 4, const_cast<void *>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

}  // namespace bi

using namespace bi;

namespace {
constexpr int64_t kI32Max = 0x7FFFFFFF;
int32_t g_last_bounds_line = 0;   // of the last bi_device_status that reported BI_ERR_BOUNDS
inline cudaStream_t as_stream(bi_stream s) { return static_cast<cudaStream_t>(s); }
}  // namespace

extern "C" {

bi_status bi_gemm_bf16(const void *X, int64_t ldx, const void *W, int64_t ldw, void *Y, int64_t ldy, int64_t M,
                       int64_t N, int64_t K, bi_stream stream) {
    if (M < 0 || N < 0 || K <= 0 || M >= kI32Max || N >= kI32Max || K >= kI32Max) return BI_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BI_OK;
    if (!X || !W || !Y) return BI_ERR_INVALID_ARG;
    if (ldx < K || ldw < K || ldy < N) return BI_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (ldx % 8 != 0 || ldw % 8 != 0 || ldy % 8 != 0 || !aligned16(X) || !aligned16(W) || !aligned16(Y))
        return BI_ERR_MISALIGNED;
    return launch_gemm_bf16(X, ldx, W, ldw, Y, ldy, M, N, K, as_stream(stream));
}

bi_status bi_grouped_gemm_bf16(const void *X, const void *W, void *Y, const int32_t *expert_offsets, int32_t E,
                               int64_t rows, int64_t N, int64_t K, bi_stream stream) {
    if (E < 1 || E > 1024 || rows < 0 || N < 0 || K <= 0 || rows >= kI32Max || K >= kI32Max ||
        static_cast<int64_t>(E) * N >= kI32Max)
        return BI_ERR_INVALID_ARG;
    if (rows == 0 || N == 0) return BI_OK;
    if (!X || !W || !Y || !expert_offsets) return BI_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return BI_ERR_MISALIGNED;
    return launch_grouped_gemm_bf16(X, W, Y, expert_offsets, E, rows, N, K, as_stream(stream));
}

bi_status bi_grouped_gemm_silu_bf16(const void *X, const void *W, void *act, const int32_t *expert_offsets, int32_t E,
                                    int64_t rows, int64_t I, int64_t K, bi_stream stream) {
    if (E < 1 || E > 1024 || rows < 0 || I < 0 || K <= 0 || rows >= kI32Max || K >= kI32Max ||
        2 * static_cast<int64_t>(E) * I >= kI32Max)
        return BI_ERR_INVALID_ARG;
    if (rows == 0 || I == 0) return BI_OK;
    if (!X || !W || !act || !expert_offsets) return BI_ERR_INVALID_ARG;
    if (K % 8 != 0 || I % 128 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(W) || !aligned16(act) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return BI_ERR_MISALIGNED;
    return launch_grouped_gemm_silu_bf16(X, W, act, expert_offsets, E, rows, I, K, as_stream(stream));
}

bi_status bi_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B, const uint8_t *B_sf, float alpha,
                        void *Y, int64_t M, int64_t N, int64_t K, bi_stream stream) {
    if (M < 0 || N < 0 || K <= 0 || M >= kI32Max || N >= kI32Max || K >= kI32Max) return BI_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return BI_OK;
    if (!A || !A_sf || !B || !B_sf || !Y) return BI_ERR_INVALID_ARG;
    if (K % 64 != 0 || N % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(A_sf) || !aligned16(B) || !aligned16(B_sf) || !aligned16(Y))
        return BI_ERR_MISALIGNED;
    return launch_gemm_nvfp4(A, A_sf, B, B_sf, alpha, Y, M, N, K, as_stream(stream));
}

bi_status bi_quantize_nvfp4(const void *X, int64_t ldx, float global_scale, uint8_t *Q, uint8_t *Q_sf, int64_t M,
                            int64_t K, bi_stream stream) {
    if (M < 0 || K <= 0 || M >= kI32Max || K >= kI32Max || !(global_scale > 0.0f) || !(global_scale <= 0x1p64f))
        return BI_ERR_INVALID_ARG;
    if (M == 0) return BI_OK;
    if (!X || !Q || !Q_sf || ldx < K) return BI_ERR_INVALID_ARG;
    if (K % 64 != 0) return BI_ERR_UNSUPPORTED;
    if (ldx % 8 != 0 || !aligned16(X) || !aligned16(Q) || !aligned16(Q_sf)) return BI_ERR_MISALIGNED;
    return launch_quantize_nvfp4(X, ldx, global_scale, Q, Q_sf, M, K, as_stream(stream));
}

namespace {
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bi_status require_device() {
    int dev;
    const DeviceInfo *info;
    return current_device(&dev, &info);
}
}  // namespace

bi_status bi_moe_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t k, int32_t renormalize,
                              int32_t *topk_ids, float *topk_weights, bi_stream stream) {
    if (T < 0 || T >= kI32Max || E < 1 || E > 1024 || k < 1 || k > 32 || k > E) return BI_ERR_INVALID_ARG;
    if (T == 0) return BI_OK;
    if (!logits || !topk_ids || !topk_weights) return BI_ERR_INVALID_ARG;
    if (!aligned4(logits) || !aligned4(topk_ids) || !aligned4(topk_weights)) return BI_ERR_MISALIGNED;
    bi_status st = require_device();
    if (st != BI_OK) return st;
    return launch_moe_topk_softmax(logits, T, E, k, renormalize, topk_ids, topk_weights, as_stream(stream));
}

bi_status bi_moe_align(const int32_t *topk_ids, int64_t T, int32_t k, int32_t E, int32_t *expert_offsets,
                       int32_t *row_token, int32_t *pos, bi_stream stream) {
    if (T < 0 || T >= kI32Max || k < 1 || E < 1 || E > 1024 || T * k >= kI32Max) return BI_ERR_INVALID_ARG;
    if (!topk_ids || !expert_offsets || !row_token || !pos) return BI_ERR_INVALID_ARG;
    if (!aligned4(topk_ids) || !aligned4(expert_offsets) || !aligned4(row_token) || !aligned4(pos))
        return BI_ERR_MISALIGNED;
    return launch_moe_align(topk_ids, T, k, E, expert_offsets, row_token, pos, as_stream(stream));
}

bi_status bi_moe_gather(const void *hidden, int64_t T, int64_t H, const int32_t *row_token, int64_t rows,
                        void *X_sorted, bi_stream stream) {
    if (T < 0 || H < 8 || rows < 0 || rows >= kI32Max) return BI_ERR_INVALID_ARG;
    if (rows == 0) return BI_OK;
    if (!hidden || !row_token || !X_sorted) return BI_ERR_INVALID_ARG;
    if (H % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(X_sorted) || !aligned4(row_token)) return BI_ERR_MISALIGNED;
    return launch_moe_gather(hidden, T, H, row_token, rows, X_sorted, as_stream(stream));
}

bi_status bi_silu_mul(const void *gate_up, int64_t rows, int64_t I, void *act, bi_stream stream) {
    if (rows < 0 || I < 8) return BI_ERR_INVALID_ARG;
    if (rows == 0) return BI_OK;
    if (!gate_up || !act) return BI_ERR_INVALID_ARG;
    if (I % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(gate_up) || !aligned16(act)) return BI_ERR_MISALIGNED;
    return launch_silu_mul(gate_up, rows, I, act, as_stream(stream));
}

bi_status bi_moe_combine(const void *Y_sorted, int64_t rows, const int32_t *pos, const float *topk_weights,
                         int64_t T, int32_t k, int64_t H, void *out, bi_stream stream) {
    if (rows < 0 || T < 0 || T >= kI32Max || k < 1 || H < 8) return BI_ERR_INVALID_ARG;
    if (T == 0) return BI_OK;
    if (!Y_sorted || !pos || !topk_weights || !out) return BI_ERR_INVALID_ARG;
    if (H % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(Y_sorted) || !aligned16(out) || !aligned4(pos) || !aligned4(topk_weights)) return BI_ERR_MISALIGNED;
    bi_status st = require_device();
    if (st != BI_OK) return st;
    return launch_moe_combine(Y_sorted, rows, pos, topk_weights, T, k, H, out, as_stream(stream));
}

bi_status bi_rmsnorm(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H, float eps,
                     bi_stream stream) {
    if (M < 0 || M >= kI32Max || H < 8 || H > 65536 || !(eps >= 0.0f)) return BI_ERR_INVALID_ARG;
    if (M == 0) return BI_OK;
    if (!x || !w || !out) return BI_ERR_INVALID_ARG;
    if (H % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (residual && !aligned16(residual)))
        return BI_ERR_MISALIGNED;
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    return launch_rmsnorm(x, residual, w, out, M, H, eps, as_stream(stream));
}

bi_status bi_rank_sum_rmsnorm(const void *const *parts, int32_t R, void *residual, const void *w, void *sum_out,
                              void *out, int64_t M, int64_t H, float eps, bi_stream stream) {
    if (R < 1 || R > 16 || M < 0 || M >= kI32Max || H < 8 || H > 65536 || !(eps >= 0.0f)) return BI_ERR_INVALID_ARG;
    if (M == 0) return BI_OK;
    if (!parts || !w || !out) return BI_ERR_INVALID_ARG;
    for (int r = 0; r < R; ++r) {
        if (!parts[r]) return BI_ERR_INVALID_ARG;
        if (!aligned16(parts[r])) return BI_ERR_MISALIGNED;
    }
    if (H % 8 != 0) return BI_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(out) || (residual && !aligned16(residual)) || (sum_out && !aligned16(sum_out)))
        return BI_ERR_MISALIGNED;
    bi_status st = require_device();
    if (st != BI_OK) return st;
    return launch_rank_sum_rmsnorm(parts, R, residual, w, sum_out, out, M, H, eps, as_stream(stream));
}

int64_t bi_attention_decode_workspace_size(int64_t B, int32_t Hq, int32_t max_seq_len) {
    if (B < 0 || Hq < 1 || max_seq_len < 1 || max_seq_len > BI_ATTENTION_MAX_SEQ_LEN) return -1;
    return attention_decode_workspace_bytes(B, Hq, max_seq_len);
}

bi_status bi_attention_decode(const void *Q, const void *K_cache, const void *V_cache, const int32_t *block_table,
                              int32_t max_blocks_per_seq, int64_t num_blocks, const int32_t *seq_lens, int64_t B,
                              int32_t Hq, int32_t Hkv, int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                              float scale, void *workspace, int64_t workspace_bytes, void *O, bi_stream stream) {
    if (B < 0 || B > 65535 || Hq < 1 || Hkv < 1 || block_size < 1 || max_seq_len < 1 ||
        max_seq_len > BI_ATTENTION_MAX_SEQ_LEN || max_blocks_per_seq < 1 || num_blocks < 1 || !(scale == scale))
        return BI_ERR_INVALID_ARG;
    if (B == 0) return BI_OK;
    if (!Q || !K_cache || !V_cache || !block_table || !seq_lens || !workspace || !O) return BI_ERR_INVALID_ARG;
    if (head_dim != 128 || Hq % Hkv != 0) return BI_ERR_UNSUPPORTED;
    const int32_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return BI_ERR_UNSUPPORTED;
    const int64_t need = attention_decode_workspace_bytes(B, Hq, max_seq_len);
    if (need < 0 || workspace_bytes < need) return BI_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K_cache) || !aligned16(V_cache) || !aligned16(O) || !aligned16(workspace) ||
        !aligned4(block_table) || !aligned4(seq_lens))
        return BI_ERR_MISALIGNED;
    bi_status st = require_device();
    if (st != BI_OK) return st;
    return launch_attention_decode(Q, K_cache, V_cache, block_table, max_blocks_per_seq, num_blocks, seq_lens, B, Hq,
                                   Hkv, head_dim, block_size, max_seq_len, scale, workspace, O, as_stream(stream));
}

bi_status bi_attention_extend(const void *Q, const int32_t *cu_q, int32_t total_q, const void *K_cache,
                              const void *V_cache, const int32_t *block_table, int32_t max_blocks_per_seq,
                              int64_t num_blocks, const int32_t *seq_lens, int64_t B, int32_t Hq, int32_t Hkv,
                              int32_t head_dim, int32_t block_size, int32_t max_seq_len, int32_t max_q_len, float scale,
                              void *O, bi_stream stream) {
    if (B < 0 || B > 65535 || total_q < 0 || Hq < 1 || Hkv < 1 || block_size < 1 || max_seq_len < 1 ||
        max_seq_len > BI_ATTENTION_MAX_SEQ_LEN || max_q_len < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        !(scale == scale))
        return BI_ERR_INVALID_ARG;
    if (B == 0 || total_q == 0) return BI_OK;
    if (!Q || !cu_q || !K_cache || !V_cache || !block_table || !seq_lens || !O) return BI_ERR_INVALID_ARG;
    if (head_dim != 128 || Hq % Hkv != 0) return BI_ERR_UNSUPPORTED;
    const int32_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return BI_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K_cache) || !aligned16(V_cache) || !aligned16(O) || !aligned4(block_table) ||
        !aligned4(seq_lens) || !aligned4(cu_q))
        return BI_ERR_MISALIGNED;
    bi_status st = require_device();
    if (st != BI_OK) return st;
    return launch_attention_extend(Q, cu_q, total_q, K_cache, V_cache, block_table, max_blocks_per_seq, num_blocks,
                                   seq_lens, B, Hq, Hkv, block_size, max_seq_len, max_q_len, scale, O,
                                   as_stream(stream));
}

bi_status bi_plan(int32_t op, int64_t M, int64_t N, int64_t K, int32_t num_sms, bi_plan_t *out) {
    if (!out || M < 0 || N < 0 || K < 0 || num_sms < 0) return BI_ERR_INVALID_ARG;
    int sms = num_sms;
    if (sms == 0) {
        int dev;
        const DeviceInfo *info;
        bi_status st = current_device(&dev, &info);
        if (st != BI_OK) return st;
        sms = info->sm_count;
    }
    std::memset(out, 0, sizeof(*out));
    switch (op) {
        case BI_OP_GEMM_BF16: plan_gemm_bf16(M, N, K, sms, out); return BI_OK;
        case BI_OP_GROUPED_GEMM_BF16: plan_grouped_gemm_bf16(M, N, K, sms, out); return BI_OK;
        case BI_OP_GROUPED_GEMM_SILU_BF16:
            plan_grouped_gemm_bf16(M, 2 * N, K, sms, out);   /* the tiles of the 2I-wide gate_up product */
            out->op = BI_OP_GROUPED_GEMM_SILU_BF16;
            return BI_OK;
        case BI_OP_GEMM_NVFP4: plan_gemm_nvfp4(M, N, K, nvfp4_clusters(sms), out); return BI_OK;
        case BI_OP_QUANTIZE_NVFP4:
            out->op = BI_OP_QUANTIZE_NVFP4;
            out->block_m = 1; out->block_n = 16; out->block_k = 16;   /* one 16-element scale block per thread */
            out->k_steps = static_cast<int32_t>(K / 16);
            out->split_k = 1; out->stages = 1; out->threads = 256;
            out->tiles_m = M; out->tiles_n = K / 16;
            {
                const int64_t g = (M * (K / 16) + 255) / 256, cap = static_cast<int64_t>(sms) * 16;
                out->grid = static_cast<int32_t>(g < cap ? g : cap);
            }
            return BI_OK;   /* N unused, K = columns */
        case BI_OP_RMSNORM: plan_rmsnorm(M, N, out); return BI_OK;   /* N carries H */
        default: return BI_ERR_INVALID_ARG;
    }
}

bi_status bi_device_status(bi_stream stream) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return BI_ERR_CUDA;
    unsigned word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof word) != cudaSuccess) return BI_ERR_CUDA;
    if (word && cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) return BI_ERR_CUDA;
    g_last_bounds_line = (word & kDevBounds) ? static_cast<int32_t>(word >> 16) : 0;
    if (word & kDevTimeout) return BI_ERR_TIMEOUT;
    if (word & kDevBounds) return BI_ERR_BOUNDS;
    if (word & kDevBadOffsets) return BI_ERR_INVALID_ARG;
    return BI_OK;
}

int32_t bi_debug_build(void) { return kDebugBuild ? 1 : 0; }

int32_t bi_last_bounds_line(void) { return g_last_bounds_line; }

bi_status bi_check_bounds(int32_t index, int32_t limit, bi_stream stream) {
    if (limit < 1 || limit > 64 || index < 0 || index > 63) return BI_ERR_INVALID_ARG;
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    return launch_bounds_check(index, limit, as_stream(stream));
}

bi_status bi_check_wait_timeout(uint32_t limit_us, bi_stream stream) {
    if (limit_us < 1 || limit_us > 2000000) return BI_ERR_INVALID_ARG;
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    return launch_wait_timeout_check(limit_us, as_stream(stream));
}

const char *bi_status_string(bi_status s) {
    switch (s) {
        case BI_OK: return "BI_OK";
        case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
        case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED";
        case BI_ERR_MISALIGNED: return "BI_ERR_MISALIGNED";
        case BI_ERR_ARCH: return "BI_ERR_ARCH";
        case BI_ERR_CUDA: return "BI_ERR_CUDA";
        case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT";
        case BI_ERR_BOUNDS: return "BI_ERR_BOUNDS";
        default: return "BI_ERR_UNKNOWN";
    }
}

int32_t bi_version(void) { return 100; }

}  // extern "C"
