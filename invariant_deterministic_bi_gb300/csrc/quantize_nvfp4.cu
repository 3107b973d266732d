// quantize_nvfp4.cu -- NVFP4 quantisation of bf16 activations (row-local, batch-invariant).
//
// The activation quantiser that feeds the NVFP4 linear layer in vLLM PR #39912
// ("NVFP4 CUTLASS batch invariant mode", test code: scaled_fp4_quant with the
// tensor's global scale). Per row and 16-element block, with global scale gs:
//   s = e4m3( amax * gs / 6 )          round to nearest even, saturating at 448
//   q = e2m1( x * gs / value(s) )      round to nearest even, saturating at 6; q = 0 if value(s) = 0
// on the exact values. Each quotient is bracketed in binary32: a lower bound
// (amax * gs times 1/6 rounded down, x times a lower bound of gs / value(s),
// each product rounded toward zero) and an upper bound (the same rounded away
// from zero), both converted with round-to-nearest-even. Rounding to a code
// is monotone, so when the two codes agree the exact value has that code too.
// When they differ (the exact value lies within a few binary32 ulps of the
// midpoint between two codes, or on it: about 1 % of elements on N(0,1) data)
// the side is decided exactly: the midpoint m times value(s) (or times 6) is
// exact in binary32, and fma(|x|, gs, -m * value(s)) has the sign of the exact
// difference; zero means a tie, which goes to the even code.
// Every output depends only on its own row and gs, so a row quantises to the
// same bytes whatever the batch. Zero magnitudes are stored as code 0 (never
// the negative-zero code 8).
//
// One thread per 16-element block, a CTA per row at a time (two rows per
// step): a warp reads 1 KB of consecutive elements (two 16-byte loads per
// thread) and writes 256 consecutive bytes of packed codes; each thread stores
// its scale byte straight into the interleaved 128x4 scale layout
// bi_gemm_nvfp4 reads.
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
    return out;
}

// 1/6 rounded down and up to binary32.
constexpr float kSixthDn = 0.166666656732559204f;   // 0x3E2AAAAA
constexpr float kSixthUp = 0.166666671633720398f;   // 0x3E2AAAAB
// 1 - 2^-21 and 1 + 2^-21: widen a quotient within 2 ulps (2^-23 relatively)
// of the exact one into bounds.
constexpr float kShrink = 0.99999952316284179688f;
constexpr float kGrow = 1.00000047683715820312f;
// Four times the midpoint between e2m1 magnitude codes a and a + 1, for
// a = 0..6 (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6): 1, 3, 5, 7, 10, 14, 20,
// one byte each.
constexpr unsigned long long kMid4 = 0x00140E0A07050301ull;

// Of the neighbouring codes lo and lo + 1, the one the exact value a * gs / d
// rounds to, given md = m * d exactly (m the midpoint of their values): the
// sign of fma(a, gs, -md) is the sign of the exact difference a*gs - m*d, and
// zero is a tie, which takes the even code.
__device__ __forceinline__ uint32_t decide(float a, float gs, float md, uint32_t lo) {
    const float diff = fmaf(a, gs, -md);
    return (diff > 0.0f || (diff == 0.0f && (lo & 1u))) ? lo + 1u : lo;
}

__global__ void __launch_bounds__(kThreads)
quantize_nvfp4_kernel(const uint4 *__restrict__ X, int64_t ldx_vec, uint8_t *__restrict__ Q, uint8_t *__restrict__ SF,
                      int M, int K, float gs, unsigned *status) {
    grid_dep_wait();      // earlier work of the stream is complete and visible
    grid_dep_launch();
    const int blocks = K / 16;                       // 16-element scale blocks per row
    const int atoms = K / 64;                        // 512-byte scale atoms per 128-row group
    // rows over the grid, a row's blocks over the CTA's threads (no 64-bit
    // division per block); two rows per step, so one thread has two blocks in flight
    auto one = [&](int r, int c) {
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
        // block scale: amax * gs / 6 bracketed by directed rounding
        uint32_t s = to_e4m3(__fmul_rz(__fmul_rz(amax, gs), kSixthDn));
        const uint32_t s_up = to_e4m3(__fmul_ru(__fmul_ru(amax, gs), kSixthUp));
        if (s != s_up) s = decide(amax, gs, 3.0f * (from_e4m3(s) + from_e4m3(s_up)), s);
        const float sv = from_e4m3(s);
        // x * gs / sv bracketed: the fast division is within 2 ulps of gs / sv
        // (sv is at least 2^-9), so inv * (1 -+ 2^-21), rounded outward, bound
        // it (both zero when sv is zero)
        const float inv = sv == 0.0f ? 0.0f : __fdividef(gs, sv);
        const float inv_dn = __fmul_rz(inv, kShrink), inv_up = __fmul_ru(inv, kGrow);
        const float sv4 = 0.25f * sv;
        uint32_t codes[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float lo[8], hi[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float xi = x[8 * h + i];
                lo[i] = __fmul_rz(xi, inv_dn);
                hi[i] = __fmul_ru(fabsf(xi), inv_up);   // magnitude only: the signs come from lo
            }
            uint32_t cl = to_e2m1x8(lo);
            const uint32_t ch = to_e2m1x8(hi);
            uint32_t dm = (cl ^ ch) & 0x77777777u;   // nibbles within a few ulps of a midpoint
            while (dm) {
                const int sh = (__ffs(dm) - 1) & ~3;          // first bit of the nibble
                dm &= ~(15u << sh);
                const int j = sh >> 3;                        // bf16 word of the element within this half
                const uint32_t wj = (j & 2) ? ((j & 1) ? w[4 * h + 3] : w[4 * h + 2]) : ((j & 1) ? w[4 * h + 1] : w[4 * h]);
                const uint32_t xb = (sh & 4) ? (wj & 0xFFFF0000u) : (wj << 16);   // odd element: high half
                const float xa = __uint_as_float(xb & 0x7FFFFFFFu);
                const uint32_t a = (cl >> sh) & 7u;
                const float m4 = static_cast<float>(static_cast<uint32_t>(kMid4 >> (8 * a)) & 0xFFu);
                const uint32_t c = decide(xa, gs, m4 * sv4, a) | ((xb >> 28) & 8u);
                cl = (cl & ~(15u << sh)) | (c << sh);
            }
            // clear the sign of every nibble whose magnitude is zero
            const uint32_t mag = cl & 0x77777777u;
            const uint32_t nz = (mag | (mag >> 1) | (mag >> 2)) & 0x11111111u;
            codes[h] = mag | (cl & (nz << 3));
        }
        *reinterpret_cast<uint2 *>(Q + static_cast<int64_t>(r) * (K / 2) + c * 8) = make_uint2(codes[0], codes[1]);
        const int64_t atom = static_cast<int64_t>(r >> 7) * atoms + (c >> 2);
        const int64_t at = atom * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
        // debug build: inside the interleaved scale buffer ((M rounded up to 128) x K/16 bytes)
        if (BI_IN_BOUNDS(at < (static_cast<int64_t>(M) + 127) / 128 * 128 * blocks, status)) SF[at] = static_cast<uint8_t>(s);
    };
    for (int r = blockIdx.x; r < M; r += 2 * gridDim.x)
        for (int c = threadIdx.x; c < blocks; c += kThreads) {
            one(r, c);
            if (r + static_cast<int>(gridDim.x) < M) one(r + gridDim.x, c);
        }
}

}  // namespace

bi_status launch_quantize_nvfp4(const void *X, int64_t ldx, float gs, uint8_t *Q, uint8_t *Q_sf, int64_t M, int64_t K,
                                cudaStream_t s) {
    int dev;
    const DeviceInfo *info;
    bi_status st = current_device(&dev, &info);
    if (st != BI_OK) return st;
    // one row per CTA at a time; 8 CTAs of 256 threads fill an SM
    const int64_t cap = static_cast<int64_t>(info->sm_count) * 8;
    const int64_t grid = M < cap ? M : cap;
    return launch_pdl(quantize_nvfp4_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<const uint4 *>(X), ldx / 8, Q, Q_sf, static_cast<int>(M), static_cast<int>(K), gs,
                      device_status_word());
}

}  // namespace bi
