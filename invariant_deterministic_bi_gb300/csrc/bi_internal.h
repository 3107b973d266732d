// bi_internal.h -- host-side helpers shared by the libbi translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "../../include/bi.h"
#include "bi_debug.cuh"

namespace bi {

constexpr int kMaxDevices = 64;      // devices the library keeps per-device state for

// Device status codes (or-ed into the per-device status word by kernels).
constexpr unsigned kDevTimeout = 1u;      // a bounded wait ran out
constexpr unsigned kDevBadOffsets = 2u;   // MoE expert offsets were not 0 <= ... <= rows

// Per-device facts, looked up once per device.
struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    bool is_sm103 = false;
};

// Current device's info; returns BI_ERR_ARCH / BI_ERR_CUDA on failure.
bi_status current_device(int *dev, const DeviceInfo **info);

// Address of this device's status word (library-owned, one per device).
unsigned *device_status_word();

// Encode a 2-D row-major tensor map (inner dimension first).
bi_status make_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                       uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                       CUtensorMapSwizzle swizzle);

// Encode a 3-D tensor map (dims inner first; strides in bytes for dims 1 and 2).
bi_status make_tmap_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t dims[3],
                       const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle);

// Encode a 4-D tensor map (dims inner first; strides in bytes for dims 1..3).
bi_status make_tmap_4d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4], CUtensorMapSwizzle swizzle);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raise a kernel's dynamic shared-memory limit once per device. `done` is a
// per-kernel bitmask of devices already configured.
bi_status ensure_smem_attr(const void *kernel, int bytes, unsigned long long *done);

// Launch `kernel` with programmatic stream serialization: it may begin while
// the previous kernel of the stream finishes (its launch and set-up overlap
// that kernel's tail). Every libbi kernel calls grid_dep_wait() before it
// touches global memory, so stream order is kept for all data.
template <typename... KArgs, typename... Args>
inline bi_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess) return BI_OK;
    cudaGetLastError();   // reported here; do not leave it for a later, unrelated check
    return BI_ERR_CUDA;
}

// Kernel launchers (defined in the .cu files); arguments already validated.
bi_status launch_gemm_bf16(const void *X, int64_t ldx, const void *W, int64_t ldw, void *Y, int64_t ldy,
                           int64_t M, int64_t N, int64_t K, cudaStream_t s);
// The dense layer with one K segment on the grouped layer's CTA-pair kernel.
bi_status launch_gemm_bf16_one_segment(const void *X, int64_t ldx, const void *W, int64_t ldw, void *Y, int64_t ldy,
                                       int64_t M, int64_t N, int64_t K, cudaStream_t s);
bi_status launch_grouped_gemm_bf16(const void *X, const void *W, void *Y, const int32_t *offsets, int32_t E,
                                   int64_t rows, int64_t N, int64_t K, cudaStream_t s);
bi_status launch_grouped_gemm_silu_bf16(const void *X, const void *W, void *act, const int32_t *offsets, int32_t E,
                                        int64_t rows, int64_t I, int64_t K, cudaStream_t s);
bi_status launch_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B, const uint8_t *B_sf,
                            float alpha, void *Y, int64_t M, int64_t N, int64_t K, cudaStream_t s);
bi_status launch_quantize_nvfp4(const void *X, int64_t ldx, float gs, uint8_t *Q, uint8_t *Q_sf, int64_t M, int64_t K,
                                cudaStream_t s);
bi_status launch_moe_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t k, int32_t renorm, int32_t *ids,
                                  float *w, cudaStream_t s);
bi_status launch_moe_align(const int32_t *ids, int64_t T, int32_t k, int32_t E, int32_t *offsets, int32_t *row_token,
                           int32_t *pos, cudaStream_t s);
bi_status launch_moe_gather(const void *hidden, int64_t T, int64_t H, const int32_t *row_token, int64_t rows,
                            void *out, cudaStream_t s);
bi_status launch_silu_mul(const void *gate_up, int64_t rows, int64_t I, void *act, cudaStream_t s);
bi_status launch_moe_combine(const void *Y, int64_t rows, const int32_t *pos, const float *w, int64_t T, int32_t k,
                             int64_t H, void *out, cudaStream_t s);
bi_status launch_rmsnorm(const void *x, void *residual, const void *w, void *out, int64_t M, int64_t H,
                         float eps, cudaStream_t s);
bi_status launch_rank_sum_rmsnorm(const void *const *parts, int32_t R, void *residual, const void *w, void *sum_out,
                                  void *out, int64_t M, int64_t H, float eps, cudaStream_t s);
int64_t attention_decode_workspace_bytes(int64_t B, int32_t Hq, int32_t max_len);
bi_status launch_attention_decode(const void *Q, const void *K, const void *V, const int32_t *table,
                                  int32_t max_blocks, int64_t num_blocks, const int32_t *lens, int64_t B, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t bs, int32_t max_len, float scale, void *workspace,
                                  void *O, cudaStream_t s);
bi_status launch_attention_extend(const void *Q, const int32_t *cu_q, int32_t total_q, const void *K, const void *V,
                                  const int32_t *table, int32_t max_blocks, int64_t num_blocks, const int32_t *lens,
                                  int64_t B, int32_t Hq, int32_t Hkv, int32_t bs, int32_t max_len, int32_t max_q,
                                  float scale, void *O, cudaStream_t s);
bi_status launch_bounds_check(int32_t index, int32_t limit, cudaStream_t s);
bi_status launch_wait_timeout_check(uint32_t limit_us, cudaStream_t s);

// Plans (M-independent except tiles_m and grid).
void plan_gemm_bf16(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *p);
void plan_gemm_bf16_one_segment(int64_t M, int64_t N, int64_t K, int sms, bi_plan_t *p);
void plan_grouped_gemm_bf16(int64_t rows, int64_t N, int64_t K, int sms, bi_plan_t *p);
void plan_gemm_nvfp4(int64_t M, int64_t N, int64_t K, int clusters, bi_plan_t *p);
// Clusters of the NVFP4 kernel resident at once on the current device (sms / 4 if the query fails).
int nvfp4_clusters(int sms);
void plan_rmsnorm(int64_t M, int64_t H, bi_plan_t *p);

}  // namespace bi
