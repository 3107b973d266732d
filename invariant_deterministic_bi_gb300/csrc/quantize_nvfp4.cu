// quantize_nvfp4.cu -- NVFP4 quantisation of bf16 activations (row-local, batch-invariant).
//
// The activation quantiser that feeds the NVFP4 linear layer in vLLM PR #39912
// ("NVFP4 CUTLASS batch invariant mode", test code: scaled_fp4_quant with the
// tensor's global scale). Per row and 16-element block, with global scale gs:
//   s = e4m3( amax * gs / 6 )          round to nearest even, saturating at 448
//   q = e2m1( x * gs / value(s) )      round to nearest even, saturating at 6; q = 0 if value(s) = 0
// evaluated in binary32 as (amax / 6) * gs and x * (gs / value(s)): one
// division per block and one multiply per element. Each quotient carries two
// roundings (within 2^-23 of the exact value, relatively), so a code or scale
// can differ from the exact definition's only where the exact value lies
// that close to the midpoint between two codes.
// Every output depends only on its own row and gs, so a row quantises to the
// same bytes whatever the batch. Zero magnitudes are stored as code 0 (never
// the negative-zero code 8).
//
// One thread per 16-element block: a warp reads 1 KB of consecutive elements
// (two 16-byte loads per thread) and writes 256 consecutive bytes of packed
// codes; each thread stores its scale byte straight into the interleaved
// 128x4 scale layout bi_gemm_nvfp4 reads.
#include <cuda_bf16.h>

#include "bi_internal.h"
#include "bi_ptx.cuh"

namespace bi {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 -> e4m3 (satfinite, round to nearest even), one byte.
__device__ __forceinline__ uint32_t to_e4m3(float v) {
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
    return out & 0xFFu;
}

// e4m3 byte -> fp32 (exact, through f16).
__device__ __forceinline__ float from_e4m3(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// Eight fp32 -> eight e2m1 nibbles (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t to_e2m1x8(const float (&y)[8]) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
    // clear the sign of every nibble whose magnitude is zero
    const uint32_t mag = out & 0x77777777u;
    const uint32_t nz = (mag | (mag >> 1) | (mag >> 2)) & 0x11111111u;
    return mag | (out & (nz << 3));
}

__global__ void __launch_bounds__(kThreads)
quantize_nvfp4_kernel(const uint4 *__restrict__ X, int64_t ldx_vec, uint8_t *__restrict__ Q, uint8_t *__restrict__ SF,
                      int64_t M, int K, float gs) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    const int blocks = K / 16;                       // 16-element scale blocks per row
    const int atoms = K / 64;                        // 512-byte scale atoms per 128-row group
    const int64_t total = M * blocks;
    for (int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; gid < total;
         gid += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t r = gid / blocks;
        const int c = static_cast<int>(gid - r * blocks);
        const uint4 *src = X + r * ldx_vec + c * 2;
        const uint4 v0 = __ldcs(src), v1 = __ldcs(src + 1);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float x[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf_lo(w[i]);
            x[2 * i + 1] = bf_hi(w[i]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
        const uint32_t s = to_e4m3(__fmul_rn(__fdiv_rn(amax, 6.0f), gs));
        const float sv = from_e4m3(s);
        const float inv = sv == 0.0f ? 0.0f : __fdiv_rn(gs, sv);    // one division per block
        uint32_t codes[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(x[8 * h + i], inv);
            codes[h] = to_e2m1x8(y);
        }
        *reinterpret_cast<uint2 *>(Q + r * (K / 2) + c * 8) = make_uint2(codes[0], codes[1]);
        const int64_t atom = (r / 128) * atoms + c / 4;
        SF[atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4] = static_cast<uint8_t>(s);
    }
}

}  // namespace

bi_status launch_quantize_nvfp4(const void *X, int64_t ldx, float gs, uint8_t *Q, uint8_t *Q_sf, int64_t M, int64_t K,
                                cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    const int64_t threads = M * (K / 16);
    int64_t grid = (threads + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(info->sm_count) * 16;
    if (grid > cap) grid = cap;
    return launch_pdl(quantize_nvfp4_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<const uint4 *>(X), ldx / 8, Q, Q_sf, M, static_cast<int>(K), gs);
}

}  // namespace bi
