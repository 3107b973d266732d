/*
 * bi.h -- libbi: batch-invariant linear layers and RMSNorm for NVIDIA GB300 (sm_103a).
 *
 * Batch invariance (vllm-ascend "Batch Invariance" guide, introduction): the
 * output for one request must not depend on how many other requests share the
 * batch or on their order. For a linear layer that means every output element
 * Y[i][j] is the same fp32 sum over k, in the same order, whatever the row
 * count M, the row's position in the batch and whatever padding rows sit next
 * to it. libbi gets there by construction:
 *   - one tile shape, one MMA instruction shape and one K loop per (N, K):
 *     nothing is chosen from M (vLLM PR #39912, "NVFP4 CUTLASS batch invariant
 *     mode", fixes its tile scheduler for the same reason);
 *   - no split-K, no stream-K, no atomics: each output element is reduced by
 *     one CTA in ascending K order;
 *   - the RMSNorm reduces each row over a fixed tree that depends only on H.
 * There is no mode switch and no fallback path: every call is invariant, and
 * an unsupported argument is an error, never a silent slower path.
 *
 * Conventions (all entry points):
 *  - Pointers are DEVICE pointers owned by the caller, 16-byte aligned; leading
 *    dimensions are in elements and must keep every row 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous on it; argument errors are returned synchronously before
 *    anything is launched; a failed launch returns BI_ERR_CUDA. Kernels are
 *    launched with programmatic stream serialization: one may begin its
 *    set-up while the previous kernel of the stream finishes, but touches no
 *    global memory before that kernel has completed, so stream order holds
 *    for all data (also inside CUDA graphs captured from the stream).
 *  - libbi allocates no device memory per call and never synchronises inside
 *    a compute call. It owns one status word per device, set by kernels whose
 *    bounded waits ran out or that found invalid device-side data
 *    (bi_device_status reads and clears it).
 *  - Empty work (M == 0, rows == 0, N == 0) returns BI_OK and launches nothing.
 *  - The current CUDA device must be an sm_103 GPU, else BI_ERR_ARCH.
 */
#ifndef LIBBI_BI_H
#define LIBBI_BI_H

#include <stdint.h>

#if defined(__GNUC__)
#define BI_API __attribute__((visibility("default")))
#else
#define BI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad offsets (host or device side) */
    BI_ERR_UNSUPPORTED = 2,   /* a size outside what the kernels handle (e.g. K % 8 != 0) */
    BI_ERR_MISALIGNED = 3,    /* pointer or leading dimension not 16-byte aligned */
    BI_ERR_ARCH = 4,          /* current device is not sm_103 */
    BI_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
    BI_ERR_TIMEOUT = 6,       /* a kernel's bounded wait ran out; its output is not valid */
    BI_ERR_BOUNDS = 7         /* debug build only: a bounds check failed and its access was skipped */
} bi_status;

/* Opaque CUDA stream handle (cudaStream_t). */
typedef void *bi_stream;

/*
 * bi_gemm_bf16 -- batch-invariant linear layer  Y = X W^T.
 *
 * The batch-invariant bf16 linear layer of the vLLM batch-invariance tracking
 * issue (#27433, "Basic framework"); row i of Y equals what a call with that
 * row alone returns, bit for bit (vLLM PR #39912, test
 * test_nvfp4_gemm_batch_invariance, states the same property for NVFP4).
 *
 *   X  bf16 [M][ldx]  row-major activations (first K columns used)
 *   W  bf16 [N][ldw]  row-major weights, nn.Linear layout (first K columns used)
 *   Y  bf16 [M][ldy]  output, first N columns written; RNE from the fp32 sum
 *
 * The fp32 reduction over k is fixed by (N, K) alone: K is cut into S
 * segments of whole 64-wide steps (S in 1..4, reported as split_k by
 * bi_plan; steps [s*T/S, (s+1)*T/S) of T = ceil(K/64)); each segment is summed
 * in ascending 16-element MMA steps from zero, and the segment sums are added
 * in segment order:
 *   Y[i][j] = bf16( P_0 + P_1 + ... + P_{S-1} ),  P_s = sum_{k in segment s} X[i][k] * W[j][k]
 * No part of this depends on M, on the row's position or on the other rows
 * (with few rows the segments run on different SMs and the sums travel
 * between them; that changes no operation).
 *
 * Requirements: M >= 0, N >= 0, K > 0; K % 8 == 0; N % 8 == 0; ldx, ldw, ldy
 * multiples of 8 and >= K (ldy >= N); M, N, K < 2^31. Y must not overlap X or W.
 */
BI_API bi_status bi_gemm_bf16(const void *X, int64_t ldx, const void *W, int64_t ldw,
                       void *Y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                       bi_stream stream);

/*
 * bi_grouped_gemm_bf16 -- batch-invariant MoE expert linear layers.
 *
 * For the MoE models the pages list as tested (Qwen3-30B-A3B, Qwen3-235B-A22B;
 * vllm-ascend guide, Tested Models): rows are grouped by expert, and rows
 * offsets[e] .. offsets[e+1]-1 of X are multiplied by expert e's weight:
 *   Y[r][j] = bf16( sum_k X[r][k] * W[e][j][k] ),  k in ascending 16-element MMA
 * steps from zero in one fp32 sum (bi_gemm_bf16's order when its plan has one
 * segment), so a token's expert output does not depend on which tokens share
 * its expert.
 *
 *   X        bf16 [rows][K]     expert-sorted activations (dense, ld = K)
 *   W        bf16 [E][N][K]     expert weights (dense)
 *   Y        bf16 [rows][N]     output (dense, ld = N)
 *   expert_offsets  int32 [E+1] DEVICE array: 0 = offsets[0] <= ... <= offsets[E] = rows
 *
 * The offsets are read on the device (no host synchronisation). If they are
 * not a non-decreasing sequence from 0 to `rows`, nothing is written and the
 * device status becomes BI_ERR_INVALID_ARG (see bi_device_status).
 * Requirements: 1 <= E <= 1024; K % 8 == 0; N % 8 == 0; E*N < 2^31.
 */
BI_API bi_status bi_grouped_gemm_bf16(const void *X, const void *W, void *Y,
                               const int32_t *expert_offsets, int32_t E, int64_t rows,
                               int64_t N, int64_t K, bi_stream stream);

/*
 * bi_grouped_gemm_silu_bf16 -- the MoE gate_up expert linear with the SiLU-mul
 * of the layer (bi_silu_mul) applied in its epilogue.
 *
 * For row r of expert e:  g = bf16(X[r] W[e][j]^T), u = bf16(X[r] W[e][I + j]^T)
 * (each exactly as bi_grouped_gemm_bf16 computes it) and
 *   act[r][j] = bf16( silu(g) * u ),  silu(g) computed as bi_silu_mul does,
 * so the result equals bi_grouped_gemm_bf16 (N = 2I) followed by bi_silu_mul,
 * bit for bit, without writing and re-reading the [rows][2I] intermediate.
 * The pages' MoE layers (vllm-ascend guide, Tested Models) have no fused
 * counterpart; this is the same layer with one pass over memory fewer.
 *
 *   X        bf16 [rows][K]     expert-sorted activations (dense, ld = K)
 *   W        bf16 [E][2I][K]    per expert: I gate rows, then I up rows (dense)
 *   act      bf16 [rows][I]     output (dense, ld = I)
 *   expert_offsets  as for bi_grouped_gemm_bf16 (same checks, same status)
 * Requirements: 1 <= E <= 1024; K % 8 == 0; I % 128 == 0; 2*E*I < 2^31.
 */
BI_API bi_status bi_grouped_gemm_silu_bf16(const void *X, const void *W, void *act,
                                           const int32_t *expert_offsets, int32_t E, int64_t rows,
                                           int64_t I, int64_t K, bi_stream stream);

/*
 * bi_gemm_nvfp4 -- batch-invariant block-scaled NVFP4 linear layer.
 *
 * vLLM PR #39912 ("NVFP4 CUTLASS batch invariant mode"): e2m1 values packed two
 * per byte (K = 2 * packed_k), one e4m3 scale per 16 consecutive K elements,
 * per-tensor global scales folded into alpha = 1 / (gs_A * gs_B):
 *   Y[i][j] = bf16( alpha * sum_k (a[i][k] * sa[i][k/16]) * (b[j][k] * sb[j][k/16]) ), fp32 accumulate
 *
 *   A     u8 [M][K/2]  e2m1 codes, element k in byte k/2, low nibble for even k
 *   B     u8 [N][K/2]  same, weights
 *   A_sf  u8           e4m3 block scales of A in the interleaved 128x4 layout:
 *                      scale (r, c) (row r, K block c = k/16) sits at byte
 *                        ((r/128) * (C/4) + c/4) * 512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *                      C = K/16 (rounded up to a multiple of 4); the buffer holds
 *                      ceil(M/128)*128 rows (padding rows may hold anything)
 *   B_sf  u8           same layout for B (ceil(N/128)*128 rows)
 *   Y     bf16 [M][N]  output (dense, ld = N)
 * The page calls this scale layout "interleaved" without defining it; the
 * layout above is the one Blackwell block-scaled MMAs read from tensor memory.
 * Requirements: K % 64 == 0 and K >= 64; N % 8 == 0.
 */
BI_API bi_status bi_gemm_nvfp4(const uint8_t *A, const uint8_t *A_sf, const uint8_t *B,
                        const uint8_t *B_sf, float alpha, void *Y,
                        int64_t M, int64_t N, int64_t K, bi_stream stream);

/*
 * bi_quantize_nvfp4 -- NVFP4 quantisation of bf16 activations for bi_gemm_nvfp4.
 *
 * The activation quantiser of vLLM PR #39912's test (scaled_fp4_quant with
 * the tensor's global scale). Per row and 16-element block, with gs = global_scale:
 *   s = e4m3( amax * gs / 6 )         round to nearest even, saturating at 448
 *   q = e2m1( x * gs / value(s) )     round to nearest even, saturating at 6; q = 0 where value(s) = 0
 * with each quotient taken on the exact values (the codes are those of the
 * exact rational numbers, ties included, not of a binary32 evaluation).
 * A zero magnitude is stored as code 0 (never code 8). Row-local: a row's
 * codes and scales do not depend on the other rows (the global scale is an
 * input, computed once for the whole tensor as in the page's test).
 *
 *   X     bf16 [M][ldx]   activations (first K columns used)
 *   Q     u8   [M][K/2]   packed e2m1 codes, element k in byte k/2, low nibble for even k
 *   Q_sf  u8              e4m3 scales in the interleaved 128x4 layout of bi_gemm_nvfp4;
 *                         the buffer holds ceil(M/128)*128 rows, rows >= M are not written
 * Requirements: K % 64 == 0, K > 0; ldx % 8 == 0, ldx >= K; 0 < global_scale <= 2^64
 * (gs = 2688 / amax(tensor) stays below 2^64 for any tensor with amax >= 1.5e-16).
 */
BI_API bi_status bi_quantize_nvfp4(const void *X, int64_t ldx, float global_scale, uint8_t *Q, uint8_t *Q_sf,
                                   int64_t M, int64_t K, bi_stream stream);

/*
 * ---- The MoE layer around bi_grouped_gemm_bf16 (MoE models listed as tested
 * on the vllm-ascend "Batch Invariance" guide: Qwen3-30B-A3B, Qwen3-235B-A22B).
 * A layer is: bi_moe_topk_softmax -> bi_moe_align -> bi_moe_gather ->
 * bi_grouped_gemm_bf16 (gate_up) -> bi_silu_mul -> bi_grouped_gemm_bf16 (down)
 * -> bi_moe_combine. Every value a token sees is computed from that token's
 * data alone, in fixed orders, so its output does not depend on the other
 * tokens in the batch. None of these calls uses atomics for results.
 */

/*
 * bi_moe_topk_softmax -- router: for each token t, the k experts with the
 * largest logits (larger first; ties go to the lower expert index) and their
 * softmax probabilities p_e = exp(l_e - max l) / sum_j exp(l_j - max l) (fp32),
 * divided by their sum when renormalize != 0.
 *   logits        f32 [T][E]      (device)
 *   topk_ids      i32 [T][k]      output
 *   topk_weights  f32 [T][k]      output
 * Requirements: 1 <= E <= 1024, 1 <= k <= min(E, 32).
 */
BI_API bi_status bi_moe_topk_softmax(const float *logits, int64_t T, int32_t E, int32_t k, int32_t renormalize,
                                     int32_t *topk_ids, float *topk_weights, bi_stream stream);

/*
 * bi_moe_align -- group the T*k (token, rank) pairs by expert, stably by
 * token: expert_offsets[e] = number of pairs routed to experts < e (E+1
 * entries); within an expert, pairs appear in increasing token order.
 * row_token[r] = token of sorted row r (T*k entries); pos[t][i] = sorted row
 * of pair (t, i) (T*k entries). Deterministic (block scans, no atomics).
 * An id outside [0, E) is skipped and the device status becomes
 * BI_ERR_INVALID_ARG. Requirements: 1 <= E <= 1024, k >= 1, T * k < 2^31 - 1.
 */
BI_API bi_status bi_moe_align(const int32_t *topk_ids, int64_t T, int32_t k, int32_t E, int32_t *expert_offsets,
                              int32_t *row_token, int32_t *pos, bi_stream stream);

/*
 * bi_moe_gather -- X_sorted[r] = hidden[row_token[r]] for r < rows.
 *   hidden bf16 [T][H], X_sorted bf16 [rows][H] (dense); H % 8 == 0.
 * A token index outside [0, T) is skipped (status BI_ERR_INVALID_ARG).
 */
BI_API bi_status bi_moe_gather(const void *hidden, int64_t T, int64_t H, const int32_t *row_token, int64_t rows,
                               void *X_sorted, bi_stream stream);

/*
 * bi_silu_mul -- act[r][j] = bf16( silu(g) * u ), g = gate_up[r][j],
 * u = gate_up[r][I + j], silu(g) = g / (1 + exp(-g)) in fp32 with the hardware
 * exponential and fast division (a few ulp of fp32 before the bf16 rounding).
 *   gate_up bf16 [rows][2I] ([gate | up]), act bf16 [rows][I]; I % 8 == 0.
 */
BI_API bi_status bi_silu_mul(const void *gate_up, int64_t rows, int64_t I, void *act, bi_stream stream);

/*
 * bi_moe_combine -- out[t] = bf16( sum_{i=0}^{k-1} w[t][i] * Y_sorted[pos[t][i]] ),
 * fp32 fused multiply-adds in top-k rank order i = 0, 1, ..., k-1.
 *   Y_sorted bf16 [rows][H], pos i32 [T][k], topk_weights f32 [T][k], out bf16 [T][H].
 * A row index outside [0, rows) is skipped (status BI_ERR_INVALID_ARG). H % 8 == 0.
 */
BI_API bi_status bi_moe_combine(const void *Y_sorted, int64_t rows, const int32_t *pos, const float *topk_weights,
                                int64_t T, int32_t k, int64_t H, void *out, bi_stream stream);

/*
 * bi_rmsnorm -- RMSNorm with optional residual add and a fixed reduction tree.
 *
 * The RMSNorm that vLLM fuses with the tensor-parallel all-reduce (vLLM PR
 * #51292, Purpose and root-cause discussion: its fused kernel reduces with
 * shuffles and block reductions whose order varies run to run). Here each row
 * is reduced by one CTA over a fixed tree that depends only on H: every thread
 * sums the squares of its elements in index order, a fixed xor-shuffle
 * butterfly combines each warp's 32 sums, and the warp sums are added in warp
 * order.
 *   h = residual ? bf16(x + residual) : x       (written back to residual)
 *   out = bf16( h * (1 / sqrt(sum(h^2)/H + eps)) * w ),  fp32 arithmetic
 *
 *   x        bf16 [M][H]      input (dense)
 *   residual bf16 [M][H]      NULLABLE; when given, updated in place to h
 *   w        bf16 [H]         weight
 *   out      bf16 [M][H]      output (dense); may be the same buffer as x
 * Requirements: H % 8 == 0, 8 <= H <= 65536; eps >= 0.
 */
BI_API bi_status bi_rmsnorm(const void *x, void *residual, const void *w, void *out,
                     int64_t M, int64_t H, float eps, bi_stream stream);

/*
 * bi_rank_sum_rmsnorm -- deterministic tensor-parallel all-reduce + RMSNorm.
 *
 * vLLM PR #51292 disables its fused all-reduce + RMSNorm under batch
 * invariance because that kernel reduces in an order that varies from run to
 * run ("a fixed-order reduction ... is bitwise-stable"). Here the R ranks'
 * partial rows, all readable from the current GPU (gathered there, or peer
 * memory), are summed in rank order 0, 1, ..., R-1 in fp32 and rounded once:
 *   a   = bf16( x_0 + x_1 + ... + x_{R-1} )   (written to sum_out if given)
 *   h   = residual ? bf16(a + residual) : a    (written back to residual)
 *   out = bf16( h / sqrt(sum(h^2)/H + eps) * w ), the bi_rmsnorm tree
 * Every rank that runs this on the same R inputs gets the same bits.
 *
 *   parts     HOST array of R DEVICE pointers, each bf16 [M][H] (dense)
 *   residual  bf16 [M][H] NULLABLE, updated in place; sum_out bf16 [M][H] NULLABLE
 *   w bf16 [H]; out bf16 [M][H]
 * Requirements: 1 <= R <= 16; H % 8 == 0, 8 <= H <= 65536; eps >= 0.
 */
BI_API bi_status bi_rank_sum_rmsnorm(const void *const *parts, int32_t R, void *residual, const void *w,
                                     void *sum_out, void *out, int64_t M, int64_t H, float eps, bi_stream stream);

/*
 * bi_attention_decode -- batch-invariant decode attention over a paged KV cache.
 *
 * Batch-invariant attention is on the vLLM tracking issue's TODO list
 * (FlashInfer, TRITON_MLA, FLASHINFER_MLA) and the vllm-ascend guide ships
 * batch-invariant attention operators. One query token per sequence b and
 * query head h (KV head g = h / (Hq/Hkv)), over the sequence's seq_lens[b]
 * cached tokens; token j of sequence b sits in physical block
 * block_table[b][j / block_size] at offset j % block_size:
 *   O[b][h] = sum_j softmax_j(scale * q.k_j) v_j
 * The KV range is split into fixed 128-token chunks by position alone (never
 * by batch size); each chunk is reduced in a fixed order and the chunks are
 * merged in chunk order, so a sequence's output does not depend on the batch.
 * Arithmetic: q.k and p.v are bf16 tensor-core products with fp32
 * accumulation; the probabilities enter p.v as a bf16 high part plus a bf16
 * low part (16 significant bits); softmax statistics and the chunk merge are
 * fp32. Chunks merge in order: m' = max(m, m_c), o = o e^(m-m') + o_c e^(m_c-m'),
 * l likewise, then o / l.
 *
 *   Q         bf16 [B][Hq][128]
 *   K_cache   bf16 [num_blocks][block_size][Hkv][128]; V_cache likewise
 *   block_table int32 [B][max_blocks_per_seq]; seq_lens int32 [B] (device)
 *   workspace caller-owned device scratch of at least
 *             bi_attention_decode_workspace_size(B, Hq, max_seq_len) bytes
 *             (fp32 per-chunk partial results); contents need not be initialised
 *   O         bf16 [B][Hq][128]
 * A sequence with seq_lens outside [1, max_seq_len] (or longer than its table)
 * is skipped, a block index outside [0, num_blocks) is ignored, and the device
 * status becomes BI_ERR_INVALID_ARG.
 * Requirements: head_dim == 128; Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8};
 * 1 <= B <= 65535; block_size >= 1; 1 <= max_seq_len <= BI_ATTENTION_MAX_SEQ_LEN;
 * workspace_bytes >= bi_attention_decode_workspace_size(B, Hq, max_seq_len).
 * bi_attention_decode_workspace_size returns -1 for arguments out of range
 * (B < 0, Hq < 1, max_seq_len outside [1, BI_ATTENTION_MAX_SEQ_LEN]) or a size
 * that does not fit in an int64_t; bi_attention_decode then refuses the call
 * with BI_ERR_INVALID_ARG.
 */
#define BI_ATTENTION_MAX_SEQ_LEN (1 << 30)
BI_API int64_t bi_attention_decode_workspace_size(int64_t B, int32_t Hq, int32_t max_seq_len);
BI_API bi_status bi_attention_decode(const void *Q, const void *K_cache, const void *V_cache,
                                     const int32_t *block_table, int32_t max_blocks_per_seq, int64_t num_blocks,
                                     const int32_t *seq_lens, int64_t B, int32_t Hq, int32_t Hkv,
                                     int32_t head_dim, int32_t block_size, int32_t max_seq_len, float scale,
                                     void *workspace, int64_t workspace_bytes, void *O, bi_stream stream);

/*
 * bi_attention_extend -- batch-invariant extend (prefill) attention over a
 * paged KV cache: the new query tokens of each sequence attend causally to
 * the sequence's cache, which already holds their keys and values.
 *
 * The pages ask for batch-invariant attention backends (vLLM tracking issue
 * #27433, TODO: FlashInfer, TRITON_MLA; vllm-ascend "Batch Invariance",
 * Implementation Details: batch-invariant attention operators). With chunked
 * prefill a sequence's new tokens share a batch with other sequences' tokens
 * and are split across steps as the scheduler decides; here neither matters.
 * Query token i of sequence b (row cu_q[b] + i of Q, 0 <= i < q_len_b =
 * cu_q[b+1] - cu_q[b]) sits at position p = seq_lens[b] - q_len_b + i and sees
 * the cached tokens 0..p:
 *   O[t][h] = sum_{j <= p} softmax_j(scale * q.k_j) v_j
 * computed exactly as bi_attention_decode computes the query of a sequence
 * of length p + 1 (the same 128-token chunks by position, per-chunk
 * arithmetic and chunk-order merge), so a token's output is the same bits
 * whether it is decoded alone, prefilled in one call, prefilled in pieces of
 * any size, or batched with any other sequences.
 *
 *   Q         bf16 [total_q][Hq][128]  the new tokens of all sequences, sequence by sequence
 *   cu_q      int32 [B+1] (device)     cu_q[0] = 0, cu_q[b+1] - cu_q[b] = q_len_b, cu_q[B] <= total_q
 *   K_cache, V_cache, block_table, block_size as in bi_attention_decode
 *   seq_lens  int32 [B] (device)       cached length of each sequence, the new tokens included
 *   O         bf16 [total_q][Hq][128]  rows of the sequences' new tokens written
 * No workspace: each CTA merges its chunks in registers. A sequence whose
 * q_len or seq_lens is out of range (q_len > max_q_len, q_len > seq_lens,
 * seq_lens > max_seq_len or longer than its table, cu_q past total_q) is
 * skipped and the device status becomes BI_ERR_INVALID_ARG.
 * Requirements: head_dim == 128; Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8};
 * 1 <= B <= 65535; 1 <= max_q_len; block_size >= 1;
 * 1 <= max_seq_len <= BI_ATTENTION_MAX_SEQ_LEN.
 */
BI_API bi_status bi_attention_extend(const void *Q, const int32_t *cu_q, int32_t total_q, const void *K_cache,
                                     const void *V_cache, const int32_t *block_table, int32_t max_blocks_per_seq,
                                     int64_t num_blocks, const int32_t *seq_lens, int64_t B, int32_t Hq,
                                     int32_t Hkv, int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                     int32_t max_q_len, float scale, void *O, bi_stream stream);

/*
 * bi_attention_decode_noalloc -- bi_attention_decode for callers that cannot
 * allocate device memory. (The pages have no counterpart: this is a library
 * convenience, not part of the method.)
 *
 * Some callers cannot call cudaMalloc or hand over a workspace: code linked
 * into a host program whose allocator has already reserved all device memory,
 * or code on a latency-critical path that must not risk the device-wide
 * synchronisation an allocation can cause. This entry point takes the same
 * arguments as bi_attention_decode minus the workspace and computes the same
 * result. Its per-chunk partial results go to one fixed array of
 * BI_ATTENTION_NOALLOC_SCRATCH_BYTES (16 MiB) that the library keeps in device
 * memory, on every GPU that loads it, until the process exits.
 *  - A problem whose partial results need more than that
 *    (bi_attention_decode_workspace_size(B, Hq, max_seq_len) > 16 MiB, or -1
 *    for a size past int64_t) is refused with BI_ERR_UNSUPPORTED before
 *    anything is launched.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the array and it keeps what the last call left in it;
 *    nothing in it needs to start at zero. Calls whose kernels overlap on the
 *    GPU (for example on two streams) race on it: serialise them.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define BI_ATTENTION_NOALLOC_SCRATCH_BYTES (16u << 20)
BI_API bi_status bi_attention_decode_noalloc(const void *Q, const void *K_cache, const void *V_cache,
                                             const int32_t *block_table, int32_t max_blocks_per_seq,
                                             int64_t num_blocks, const int32_t *seq_lens, int64_t B, int32_t Hq,
                                             int32_t Hkv, int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                             float scale, void *O, bi_stream stream);

/* Operation ids for bi_plan. */
enum { BI_OP_GEMM_BF16 = 0, BI_OP_GROUPED_GEMM_BF16 = 1, BI_OP_GEMM_NVFP4 = 2, BI_OP_RMSNORM = 3,
       BI_OP_QUANTIZE_NVFP4 = 4, BI_OP_GROUPED_GEMM_SILU_BF16 = 5 /* N carries I */ };

/*
 * bi_plan -- the launch plan a call with these sizes uses (host only, no GPU needed).
 *
 * Everything that decides the arithmetic (tile, MMA shape, K step, K-step
 * count, split) depends on (N, K) or H only; tiles_m and grid also depend on M
 * (or rows). For the grouped GEMM, M is the row capacity and the real tile
 * count is decided on the device. num_sms = 0 means "the current device's SM
 * count" (then a CUDA device is needed); pass e.g. 152 to plan without one.
 */
typedef struct {
    int32_t op;
    int32_t block_m, block_n, block_k;   /* CTA tile (rows, cols, K step); RMSNorm: 1 row per CTA, H, 8 */
    int32_t mma_m, mma_n, mma_k;         /* tcgen05.mma instruction shape (0 for RMSNorm) */
    int32_t k_steps;                     /* K steps per output tile (fixed by K); RMSNorm: vectors per thread */
    int32_t split_k;                     /* bf16 GEMM: K segments S (1..4, fixed by N, K); others 1 */
    int32_t stages;                      /* shared-memory pipeline depth */
    int32_t threads;                     /* threads per CTA */
    int32_t smem_bytes;                  /* dynamic shared memory per CTA */
    int64_t tiles_m, tiles_n;            /* output tiles (tiles_m depends on M) */
    int32_t grid;                        /* CTAs launched (persistent GEMMs: <= SM count) */
    int32_t reduce_tree;                 /* RMSNorm: elements each thread sums in index order */
} bi_plan_t;

BI_API bi_status bi_plan(int32_t op, int64_t M, int64_t N, int64_t K, int32_t num_sms, bi_plan_t *out);

/*
 * bi_device_status -- synchronise `stream`, then read and clear the current
 * device's status word. Returns BI_OK, BI_ERR_TIMEOUT (a bounded wait in a
 * kernel ran out; that call's output is invalid), BI_ERR_BOUNDS (debug build:
 * a bounds check failed; bi_last_bounds_line() names its source line),
 * BI_ERR_INVALID_ARG (a kernel found invalid device-side data, e.g. MoE
 * offsets) or BI_ERR_CUDA.
 */
BI_API bi_status bi_device_status(bi_stream stream);

/*
 * bi_check_wait_timeout -- launch one CTA that waits on a shared-memory
 * barrier nobody arrives at, with a limit of `limit_us` microseconds
 * (1 .. 2,000,000), then records BI_ERR_TIMEOUT in the status word and
 * returns. Exercises the same bounded-wait path the GEMM kernels use; a
 * following bi_device_status(stream) returns BI_ERR_TIMEOUT.
 */
BI_API bi_status bi_check_wait_timeout(uint32_t limit_us, bi_stream stream);

/*
 * The debug build (libbi_debug.so, compiled with BI_DEBUG): every kernel
 * checks the indices and coordinates it computes -- TMA copy coordinates,
 * tensor-memory columns, shared-memory areas, workspace and output rows --
 * against the extents of its buffers before using them. A failed check skips
 * the access and records BI_ERR_BOUNDS in the device status word (never a
 * trap or an assert); the release build (libbi.so) compiles the checks away.
 * Outputs of the two builds are identical when no check fails.
 *
 * bi_debug_build -- 1 in the debug build, 0 in the release build.
 * bi_last_bounds_line -- the source line of the failed check that the last
 *   bi_device_status call reported (0 if none).
 * bi_check_bounds -- launch one thread that writes element `index` of a
 *   library-owned 64-element array under a bounds check against `limit`
 *   (1..64; index 0..63); in the debug build an index >= limit is skipped and
 *   recorded, so a following bi_device_status returns BI_ERR_BOUNDS. It
 *   exercises the check path without touching any caller memory.
 */
BI_API int32_t bi_debug_build(void);
BI_API int32_t bi_last_bounds_line(void);
BI_API bi_status bi_check_bounds(int32_t index, int32_t limit, bi_stream stream);

/* Human-readable name of a status code (static string). */
BI_API const char *bi_status_string(bi_status s);

/* Library version: major*10000 + minor*100 + patch. */
BI_API int32_t bi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LIBBI_BI_H */
