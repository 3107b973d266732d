/*
 * oracle.c -- plain, slow fp64 CPU oracle for the batch-invariant linear layer
 * and RMSNorm.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg
 * do. It shares no code, header, table or constant with the CUDA library.
 *
 * Every routine evaluates the plain definition of what the kernel computes, in
 * fp64, on the same stored (bf16 / e2m1 / e4m3) values the kernel reads, with
 * no blocking, fusion or reordering: loops run in index order. Rows are
 * distributed over OpenMP threads (each output element is still one
 * sequential sum), which changes nothing but wall time.
 *
 * Sources (web pages on batch invariance in vLLM serving):
 *  - Batch invariance: a request's output does not depend on batch size or
 *    on request order (vllm-ascend "Batch Invariance" guide, introduction).
 *  - Linear layer Y = X W^T over nn.Linear weights; its NVFP4 form
 *    alpha * (A_fp4 . sf_A)(B_fp4 . sf_B)^T with alpha = 1/(gs_A gs_B)
 *    (vLLM PR #39912 "NVFP4 CUTLASS batch invariant mode", test code);
 *    the dequantise-then-multiply reading is the "emulation" backend of the
 *    same PR's kernel selector.
 *  - RMSNorm after the residual add (vLLM PR #51292, fused all-reduce +
 *    RMSNorm, Purpose / root-cause discussion). The pages give no formula;
 *    the standard y = h / sqrt(mean(h^2) + eps) * w is used.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even mantissa). bf16 keeps 8
 * significant bits; its smallest exponent is that of binary32 (subnormal
 * quantum 2^-133); values past the largest finite bf16 become infinity. */
static uint16_t double_to_bf16(double v)
{
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int e;
    (void)frexp(fabs(v), &e);                  /* |v| = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;                          /* quantum of an 8-bit significand */
    if (qexp < -133) qexp = -133;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(v / q) * q;           /* default rounding: nearest, ties even */
    float f = (float)r;                        /* exact: r has <= 8 significant bits */
    if (fabs(r) > 3.3895313892515355e38) f = signbit(r) ? -INFINITY : INFINITY;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0
 * is subnormal (0 or 0.5). OCP Microscaling Formats spec, FP4 E2M1. */
static double e2m1_to_double(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - 1);
    return s ? -mag : mag;
}

/* e4m3 (FN): sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities.
 * OCP 8-bit Floating Point spec, E4M3. */
static double e4m3_to_double(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Exported decoders (used by the format pins). */
double oracle_e2m1_value(unsigned code) { return e2m1_to_double(code & 15u); }
double oracle_e4m3_value(unsigned code) { return e4m3_to_double(code & 255u); }
double oracle_bf16_value(uint16_t bits) { return bf16_to_double(bits); }
uint16_t oracle_bf16_round(double v) { return double_to_bf16(v); }

/* Round n doubles to bf16 bit patterns (same rule as double_to_bf16). */
void oracle_bf16_round_array(int64_t n, const double *v, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the parallel loops from now on (n >= 1); only for timing the
   oracle on fewer cores: every output element is one sequential sum, so the
   results do not depend on it. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Y[i][j] = sum_{k=0}^{K-1} X[i][k] * W[j][k]   (linear layer, Y = X W^T).
 * X: bf16 [M][ldx], W: bf16 [N][ldw] (nn.Linear layout), Y: fp64 [M][ldy]. */
void oracle_gemm_bf16(int64_t M, int64_t N, int64_t K,
                      const uint16_t *X, int64_t ldx,
                      const uint16_t *W, int64_t ldw,
                      double *Y, int64_t ldy)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_double(X[i * ldx + k]) * bf16_to_double(W[j * ldw + k]);
            Y[i * ldy + j] = acc;
        }
    }
}

/* Grouped (MoE expert) linear layers: rows offsets[e] .. offsets[e+1]-1 of X
 * belong to expert e and are multiplied by that expert's weight W[e] ([N][K]).
 * X: bf16 [offsets[E]][K], W: bf16 [E][N][K], Y: fp64 [offsets[E]][N]. */
void oracle_grouped_gemm_bf16(int32_t E, const int32_t *offsets, int64_t N, int64_t K,
                              const uint16_t *X, const uint16_t *W, double *Y)
{
    for (int32_t e = 0; e < E; ++e) {
        const int64_t r0 = offsets[e], r1 = offsets[e + 1];
        const uint16_t *We = W + (int64_t)e * N * K;
#pragma omp parallel for schedule(static)
        for (int64_t i = r0; i < r1; ++i) {
            for (int64_t j = 0; j < N; ++j) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += bf16_to_double(X[i * K + k]) * bf16_to_double(We[j * K + k]);
                Y[i * N + j] = acc;
            }
        }
    }
}

/* Block-scaled NVFP4 linear layer, dequantised in fp64:
 *   Y[i][j] = alpha * sum_k (a[i][k] * sa[i][k/16]) * (b[j][k] * sb[j][k/16])
 * A: packed e2m1 [M][K/2] (element k in byte k/2, low nibble for even k),
 * SA: e4m3 [M][K/16] row-major; B, SB likewise with N rows; Y fp64 [M][N]. */
void oracle_gemm_nvfp4(int64_t M, int64_t N, int64_t K,
                       const uint8_t *A, const uint8_t *SA,
                       const uint8_t *B, const uint8_t *SB,
                       double alpha, double *Y)
{
    const int64_t KB = K / 2, KS = K / 16;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                unsigned abyte = A[i * KB + k / 2], bbyte = B[j * KB + k / 2];
                unsigned ac = (k & 1) ? (abyte >> 4) : (abyte & 15u);
                unsigned bc = (k & 1) ? (bbyte >> 4) : (bbyte & 15u);
                double av = e2m1_to_double(ac) * e4m3_to_double(SA[i * KS + k / 16]);
                double bv = e2m1_to_double(bc) * e4m3_to_double(SB[j * KS + k / 16]);
                acc += av * bv;
            }
            Y[i * N + j] = alpha * acc;
        }
    }
}

/* ---- NVFP4 quantisation of activations (scaled_fp4_quant in the page's test).
 * Per row r and 16-element block b, with the per-tensor global scale gs, the
 * plain definition on exact values:
 *   amax = max |x| over the block
 *   s    = e4m3_rne_satfinite( amax * gs / 6 )
 *   q_k  = e2m1_rne( clamp( x_k * gs / value(s), -6, 6 ) ),  q = 0 if value(s) == 0
 * Both quotients are evaluated in fp64: x * gs and amax * gs are exact (a bf16
 * significand times a binary32 one has at most 32 bits) and the one division
 * rounds once, which cannot carry the quotient across a rounding boundary of
 * e4m3 or e2m1 (a boundary has at most 5 significant bits, so a quotient
 * that is not on it is at least 2^-40 away, relatively). The codes are
 * therefore those of the exact rational values.
 * Encoders are written from the format definitions: round to the nearest
 * representable value by binade (quantum 2^(e - mantissa bits)), ties to even. */

/* Round half to even of a non-negative double. */
static double rne(double v) { return nearbyint(v); }

static unsigned e4m3_encode_satfinite(double v) /* v >= 0 */
{
    if (!(v < 448.0)) return 0x7Eu;                   /* saturate (also +inf) */
    if (v < ldexp(1.0, -6)) {                         /* subnormal binade: quantum 2^-9 */
        double m = rne(v * 512.0);                    /* exact scaling by a power of two */
        return (unsigned)m;                           /* m == 8 is 2^-6, code 0x08 */
    }
    int e;
    (void)frexp(v, &e);                               /* v = f * 2^e, f in [0.5, 1) */
    e -= 1;                                           /* v in [2^e, 2^(e+1)) */
    double m = rne(ldexp(v, 3 - e));                  /* significand in [8, 16] */
    if (m == 16.0) { m = 8.0; e += 1; }
    if (e > 8) return 0x7Eu;
    return ((unsigned)(e + 7) << 3) | ((unsigned)m - 8u);
}

static unsigned e2m1_encode_mag(double a) /* 0 <= a <= 6 */
{
    if (a < 2.0) return (unsigned)rne(a * 2.0);                  /* quantum 0.5: codes 0..4 */
    if (a < 4.0) return 2u + (unsigned)rne(a);                   /* quantum 1: 2,3,4 -> codes 4,5,6 */
    return 4u + (unsigned)rne(a * 0.5);                          /* quantum 2: 2,3 -> codes 6,7 */
}

unsigned oracle_e4m3_encode(double v) { return e4m3_encode_satfinite(v); }
unsigned oracle_e2m1_encode(double v)
{
    unsigned c = e2m1_encode_mag(fmin(fabs(v), 6.0));
    return (v < 0.0 && c != 0u) ? (c | 8u) : c;
}

/* Codes of one row's blocks for given scale codes S (row-major [K/16]). */
static void encode_row(int64_t K, const uint16_t *x, double gs, const uint8_t *S, uint8_t *Q)
{
    for (int64_t b = 0; b < K / 16; ++b) {
        double sv = e4m3_to_double(S[b]);
        for (int k = 0; k < 16; k += 2) {
            unsigned c[2];
            for (int h = 0; h < 2; ++h) {
                if (sv == 0.0) { c[h] = 0u; continue; }
                double y = bf16_to_double(x[b * 16 + k + h]) * gs / sv;
                c[h] = oracle_e2m1_encode(fmin(fmax(y, -6.0), 6.0));
            }
            Q[(b * 16 + k) / 2] = (uint8_t)(c[0] | (c[1] << 4));
        }
    }
}

/* X: bf16 [M][K]; Q: packed e2m1 [M][K/2] (low nibble = even k); S: e4m3 [M][K/16]. */
void oracle_quantize_nvfp4(int64_t M, int64_t K, const uint16_t *X, float gs, uint8_t *Q, uint8_t *S)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t b = 0; b < K / 16; ++b) {
            double amax = 0.0;
            for (int k = 0; k < 16; ++k) {
                double a = fabs(bf16_to_double(X[i * K + b * 16 + k]));
                if (a > amax) amax = a;
            }
            S[i * (K / 16) + b] = (uint8_t)e4m3_encode_satfinite(amax * (double)gs / 6.0);
        }
        encode_row(K, X + i * K, (double)gs, S + i * (K / 16), Q + i * (K / 2));
    }
}

/* The codes of the definition above for given block scales S [M][K/16]
 * (used to check codes in a block whose scale was taken from elsewhere). */
void oracle_quantize_nvfp4_codes(int64_t M, int64_t K, const uint16_t *X, float gs, const uint8_t *S, uint8_t *Q)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) encode_row(K, X + i * K, (double)gs, S + i * (K / 16), Q + i * (K / 2));
}

/* ---- MoE layer surroundings (the MoE models listed as tested on the vllm-ascend
 * "Batch Invariance" guide: Qwen3-30B-A3B, Qwen3-235B-A22B).
 *
 * Routing, per token t with router logits l[t][0..E-1] (fp32):
 *   ids  = the k experts with the largest logits, larger first, ties to the
 *          lower expert index (softmax is monotonic, so these are also the
 *          k largest softmax probabilities);
 *   p_e  = exp(l_e - max l) / sum_j exp(l_j - max l)   (fp64)
 *   w_i  = p_{ids[i]}, divided by sum_i p_{ids[i]} when renormalize != 0. */
void oracle_moe_topk_softmax(int64_t T, int32_t E, int32_t k, const float *logits, int renormalize,
                             int32_t *ids, double *w)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        double mx = -INFINITY;
        for (int32_t e = 0; e < E; ++e)
            if ((double)l[e] > mx) mx = (double)l[e];
        double sum = 0.0;
        for (int32_t e = 0; e < E; ++e) sum += exp((double)l[e] - mx);
        /* selection: repeatedly take the largest remaining logit, lowest index on ties */
        unsigned char taken[4096];
        for (int32_t e = 0; e < E; ++e) taken[e] = 0;
        double wsum = 0.0;
        for (int32_t i = 0; i < k; ++i) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            ids[t * k + i] = best;
            w[t * k + i] = exp((double)l[best] - mx) / sum;
            wsum += w[t * k + i];
        }
        if (renormalize)
            for (int32_t i = 0; i < k; ++i) w[t * k + i] /= wsum;
    }
}

/* Group the T*k (token, rank) pairs by expert, stably by token:
 * offsets[e] = number of pairs with expert < e; within expert e the pairs
 * appear in increasing token order. row_token[r] = token of sorted row r,
 * pos[t][i] = sorted row of pair (t, i). */
void oracle_moe_align(int64_t T, int32_t k, int32_t E, const int32_t *ids, int32_t *offsets, int32_t *row_token,
                      int32_t *pos)
{
    for (int32_t e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t i = 0; i < k; ++i) offsets[ids[t * k + i] + 1] += 1;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (int32_t e = 0; e < E; ++e) {
        int32_t r = offsets[e];
        for (int64_t t = 0; t < T; ++t)
            for (int32_t i = 0; i < k; ++i)
                if (ids[t * k + i] == e) {
                    row_token[r] = (int32_t)t;
                    pos[t * k + i] = r;
                    ++r;
                }
    }
}

/* act[r][j] = silu(g) * u with g = gu[r][j], u = gu[r][I + j], silu(g) = g / (1 + exp(-g)). */
void oracle_silu_mul(int64_t R, int64_t I, const uint16_t *gu, double *act)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t j = 0; j < I; ++j) {
            double g = bf16_to_double(gu[r * 2 * I + j]);
            double u = bf16_to_double(gu[r * 2 * I + I + j]);
            act[r * I + j] = g / (1.0 + exp(-g)) * u;
        }
}

/* out[t][h] = sum_{i=0}^{k-1} w[t][i] * Y[pos[t][i]][h]   (rank order i = 0..k-1). */
void oracle_moe_combine(int64_t T, int32_t k, int64_t H, const uint16_t *Y, const int32_t *pos, const double *w,
                        double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t i = 0; i < k; ++i)
                acc += w[t * k + i] * bf16_to_double(Y[(int64_t)pos[t * k + i] * H + h]);
            out[t * H + h] = acc;
        }
}

/* ---- Deterministic tensor-parallel all-reduce followed by RMSNorm (the pair
 * vLLM PR #51292 stops fusing under batch invariance: "a fixed-order reduction
 * is bitwise-stable"). R ranks hold partial rows x_r; the all-reduced row is
 *   a = bf16( x_0 + x_1 + ... + x_{R-1} )     (exact sum, one rounding)
 * and then, as in oracle_rmsnorm: h = residual ? bf16(a + residual) : a,
 *   y = h / sqrt(mean(h^2) + eps) * w.
 * parts: bf16 [R][M][H]; a_out, h_out (nullable): bf16 bits; y: fp64 [M][H]. */
void oracle_rank_sum_rmsnorm(int32_t R, int64_t M, int64_t H, const uint16_t *parts, const uint16_t *residual,
                             const uint16_t *w, double eps, double *y, uint16_t *a_out, uint16_t *h_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0;
        for (int64_t k = 0; k < H; ++k) {
            double s = 0.0;
            for (int32_t r = 0; r < R; ++r) s += bf16_to_double(parts[((int64_t)r * M + i) * H + k]);
            uint16_t ab = double_to_bf16(s);
            if (a_out) a_out[i * H + k] = ab;
            double h = bf16_to_double(ab);
            if (residual) {
                uint16_t hb = double_to_bf16(h + bf16_to_double(residual[i * H + k]));
                if (h_out) h_out[i * H + k] = hb;
                h = bf16_to_double(hb);
            }
            ss += h * h;
        }
        double rinv = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t k = 0; k < H; ++k) {
            double s = 0.0;
            for (int32_t r = 0; r < R; ++r) s += bf16_to_double(parts[((int64_t)r * M + i) * H + k]);
            double h = bf16_to_double(double_to_bf16(s));
            if (residual) h = bf16_to_double(double_to_bf16(h + bf16_to_double(residual[i * H + k])));
            y[i * H + k] = h * rinv * bf16_to_double(w[k]);
        }
    }
}

/* ---- Decode attention over a paged KV cache (batch-invariant attention is on
 * the tracking issue's TODO list: FlashInfer, TRITON_MLA, FLASHINFER_MLA; the
 * vllm-ascend guide's batch-invariant attention operators).
 * For sequence b, query head h (KV head g = h / (Hq / Hkv)) and its L_b
 * cached tokens j (token j of sequence b lives in block table[b][j / bs] at
 * offset j % bs):
 *   s_j = scale * sum_d q[b][h][d] * k_j[g][d]
 *   o[b][h][d] = sum_j softmax(s)_j * v_j[g][d]          (fp64, exact softmax)
 * Q: bf16 [B][Hq][D]; K, V: bf16 [blocks][bs][Hkv][D]; table: int32 [B][max_blocks];
 * lens: int32 [B] (>= 1); O: fp64 [B][Hq][D]. */
void oracle_attention_decode(int64_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t bs, int32_t max_blocks,
                             const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *table,
                             const int32_t *lens, double scale, double *O)
{
#pragma omp parallel for schedule(static)
    for (int64_t bh = 0; bh < B * Hq; ++bh) {
        const int64_t b = bh / Hq;
        const int32_t h = (int32_t)(bh % Hq), g = h / (Hq / Hkv);
        const int32_t L = lens[b];
        double mx = -INFINITY;
        for (int32_t j = 0; j < L; ++j) {
            const int64_t blk = table[b * max_blocks + j / bs];
            const uint16_t *k = K + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d) s += bf16_to_double(Q[(b * Hq + h) * D + d]) * bf16_to_double(k[d]);
            s *= scale;
            if (s > mx) mx = s;
        }
        double den = 0.0;
        double *o = O + (b * Hq + h) * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int32_t j = 0; j < L; ++j) {
            const int64_t blk = table[b * max_blocks + j / bs];
            const uint16_t *k = K + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            const uint16_t *v = V + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d) s += bf16_to_double(Q[(b * Hq + h) * D + d]) * bf16_to_double(k[d]);
            const double p = exp(s * scale - mx);
            den += p;
            for (int32_t d = 0; d < D; ++d) o[d] += p * bf16_to_double(v[d]);
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= den;
    }
}

/* ---- Extend (prefill) attention over a paged KV cache: q_len_b new query
 * tokens of sequence b attend causally to its cache, which already holds
 * their keys and values (the decode case is q_len_b = 1). Query token i of
 * sequence b (0 <= i < q_len_b, row cu_q[b] + i of Q) sits at position
 * p = L_b - q_len_b + i of the sequence, and sees the L_b - q_len_b + i + 1
 * cached tokens j <= p:
 *   s_j = scale * sum_d q[t][h][d] * k_j[g][d]
 *   o[t][h][d] = sum_{j <= p} softmax(s)_j * v_j[g][d]     (fp64, exact softmax)
 * Q: bf16 [total_q][Hq][D]; cu_q: int32 [B+1] (cu_q[0] = 0, rows of each
 * sequence); K, V, table, lens as in oracle_attention_decode (lens = the
 * cached length including the new tokens); O: fp64 [total_q][Hq][D]. */
void oracle_attention_extend(int64_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t bs, int32_t max_blocks,
                             const uint16_t *Q, const int32_t *cu_q, const uint16_t *K, const uint16_t *V,
                             const int32_t *table, const int32_t *lens, double scale, double *O)
{
    const int64_t total_q = cu_q[B];
#pragma omp parallel for schedule(dynamic)
    for (int64_t th = 0; th < total_q * Hq; ++th) {
        const int64_t t = th / Hq;
        const int32_t h = (int32_t)(th % Hq), g = h / (Hq / Hkv);
        int64_t b = 0;
        while (cu_q[b + 1] <= t) ++b;
        const int32_t qlen = cu_q[b + 1] - cu_q[b];
        const int32_t pos = lens[b] - qlen + (int32_t)(t - cu_q[b]);
        const uint16_t *q = Q + (t * Hq + h) * D;
        double mx = -INFINITY;
        for (int32_t j = 0; j <= pos; ++j) {
            const int64_t blk = table[b * max_blocks + j / bs];
            const uint16_t *k = K + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d) s += bf16_to_double(q[d]) * bf16_to_double(k[d]);
            s *= scale;
            if (s > mx) mx = s;
        }
        double den = 0.0;
        double *o = O + (t * Hq + h) * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int32_t j = 0; j <= pos; ++j) {
            const int64_t blk = table[b * max_blocks + j / bs];
            const uint16_t *k = K + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            const uint16_t *v = V + ((blk * bs + j % bs) * (int64_t)Hkv + g) * D;
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d) s += bf16_to_double(q[d]) * bf16_to_double(k[d]);
            const double pr = exp(s * scale - mx);
            den += pr;
            for (int32_t d = 0; d < D; ++d) o[d] += pr * bf16_to_double(v[d]);
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= den;
    }
}

/* RMSNorm with optional residual add, per row i:
 *   h = residual ? bf16(x + residual) : x         (the stored, rounded sum)
 *   y = h / sqrt( (1/H) sum_k h_k^2 + eps ) * w
 * x, residual: bf16 [M][H]; w: bf16 [H]; y: fp64 [M][H];
 * h_out (nullable): bf16 bits of h, what the kernel writes back to residual. */
void oracle_rmsnorm(int64_t M, int64_t H, const uint16_t *x, const uint16_t *residual,
                    const uint16_t *w, double eps, double *y, uint16_t *h_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0;
        for (int64_t k = 0; k < H; ++k) {
            double h;
            if (residual) {
                uint16_t hb = double_to_bf16(bf16_to_double(x[i * H + k]) +
                                             bf16_to_double(residual[i * H + k]));
                if (h_out) h_out[i * H + k] = hb;
                h = bf16_to_double(hb);
            } else {
                h = bf16_to_double(x[i * H + k]);
            }
            ss += h * h;
        }
        double r = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t k = 0; k < H; ++k) {
            double h = residual ? bf16_to_double(double_to_bf16(bf16_to_double(x[i * H + k]) +
                                                                bf16_to_double(residual[i * H + k])))
                                : bf16_to_double(x[i * H + k]);
            y[i * H + k] = h * r * bf16_to_double(w[k]);
        }
    }
}
