/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused exact-attention forward library.
 *
 * Pages this interface implements (titles as published):
 *   [WGC] "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践"
 *   [JJ]  "大模型加速-核心网络算子-Flash Attention V3"
 *   [YT]  "FlashAttention V3：优化框架吞吐量的关键技术实践"
 *
 * Conventions shared by every entry point:
 *   - Tensors are caller-owned DEVICE memory on the current CUDA device, laid out
 *     [B, H, N, d] contiguous (d innermost, row stride d elements).  q, k, v, o,
 *     x and x8 must be 16-byte aligned (the kernels move them with TMA or 16-byte
 *     vectors); lse and scale arrays must be 4-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call only enqueues work on that stream: it never synchronises, never
 *     allocates device memory, and returns as soon as the launch is queued.
 *   - Errors are returned as attn_status_t; nothing is launched when a call
 *     returns anything other than ATTN_OK.  No call throws or exits.
 *   - The library keeps one device status word per GPU.  A kernel that gives up
 *     on an internal wait (ATTN_ERR_TIMEOUT) records it there; read it with
 *     attn_get_device_status().
 *   - Mask: key j is allowed for query i when 0 <= j < N and
 *       causal != 0  ->  j <= i
 *       window  > 0  ->  j >= i - window, and (when causal == 0) j <= i + window
 *     ([YT] §2.1.2 稀疏性感知的Mask优化 builds the band max(0,i-w) .. i+w; the
 *     causal band keeps its left edge).  window <= 0 means no window.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null pointer, B/H/N < 1, scale not finite and > 0 */
    ATTN_ERR_UNSUPPORTED = 2, /* head dim, block size or sequence length not supported */
    ATTN_ERR_MISALIGNED = 3,  /* a pointer breaks the alignment rule above */
    ATTN_ERR_CUDA = 4,        /* the CUDA runtime or driver reported an error */
    ATTN_ERR_TIMEOUT = 5      /* a kernel gave up on an internal wait (device status only) */
} attn_status_t;

/* FP8 formats ([JJ] §1.5 低精度FP8: E4M3, 4 exponent / 3 mantissa bits, largest 448;
 * E5M2, 5 exponent / 2 mantissa bits, largest 57344 -- wider range, less precision).
 * ATTN_FP8_E4M3_POW2: E4M3 codes whose per-block scale is a power of two. */
typedef enum { ATTN_FP8_E4M3 = 0, ATTN_FP8_E5M2 = 1, ATTN_FP8_E4M3_POW2 = 2 } attn_fp8_format_t;

/*
 * attn_fwd_bf16 -- O = softmax(scale * Q K^T + mask) V and LSE, bf16 in / bf16 out.
 *
 * [WGC] §2 GEMM-Softmax 融合流水线 and [YT] §1.2 (softmax, mask and both matmuls
 * fused in one kernel, the N x N scores never stored); [JJ] §2.1-2.2 (warp
 * specialised producer/consumer pipeline, softmax overlapped with the GEMMs).
 *
 *   q, k, v : const bf16 [B, H, N, d]
 *   o       : bf16 [B, H, N, d], written
 *   lse     : float [B, H, N], written: natural-log log-sum-exp of the masked,
 *             scaled scores of each query row
 *   B, H, N : >= 1;  d in {64, 128, 256} (else ATTN_ERR_UNSUPPORTED)
 *   scale   : finite, > 0 (typically 1/sqrt(d))
 *   causal, window : mask, see above
 * Accumulation is fp32 (scores, running max/sum, O); P is rounded to bf16 for
 * the second matmul.
 */
attn_status_t attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int N, int d, float scale, int causal, int window,
                            void* stream);

/*
 * attn_bwd_bf16 -- backward pass of attn_fwd_bf16: dQ, dK, dV for an upstream dO.
 *
 * The backward pass the pages mention for training ([YT] §2.3.2 流水线并行: forward and
 * backward of micro-batches overlapped; [JJ] §2.3-2.4 call their kernel the forward pass).
 * With P = exp(scale * Q K^T + mask - LSE) (the forward's LSE, so P is normalised):
 *     D_i = dO_i . O_i,  dP = dO V^T,  dS = P * (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO.
 *   q, k, v, o, dout : const bf16 [B, H, N, d]; o and lse as attn_fwd_bf16 wrote them
 *   lse        : const float [B, H, N] (natural log)
 *   dq, dk, dv : bf16 [B, H, N, d], written
 *   workspace  : device memory of attn_bwd_workspace_bytes(B, H, N) bytes (holds D)
 *   d in {64, 128}; scale, causal, window as the forward call that made o and lse
 * Alignment: tensors 16 bytes; lse and workspace 4 bytes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N);

/*
 * attn_bwd_bf16_varlen -- attn_bwd_bf16 over packed variable-length sequences, the
 * backward of attn_fwd_bf16_varlen ([YT] §1.1: variable sequence lengths).
 *
 * Every sequence is its own attention problem, as in the forward.
 *   q, k, v, o, dout : const bf16 [T, H, d] packed; o and lse as attn_fwd_bf16_varlen
 *                      wrote them (lse float [H, T], natural log)
 *   dq, dk, dv       : bf16 [T, H, d], written for the tokens of every sequence
 *   workspace        : device memory of at least attn_bwd_workspace_bytes(1, H, T) bytes
 *   cu_seqlens       : int32 [num_seqs + 1] on the device, as attn_fwd_bf16_varlen
 *   max_seqlen       : >= every sequence's length (sizes the work); total_tokens = T
 *   d in {64, 128}; scale, causal, window as the forward call.  T == 0 returns ATTN_OK.
 * Offsets are clamped on the device; tokens outside every sequence are not written.
 */
attn_status_t attn_bwd_bf16_varlen(const void* q, const void* k, const void* v, const void* o,
                                   const void* dout, const float* lse, void* dq, void* dk,
                                   void* dv, void* workspace, size_t workspace_bytes,
                                   const int* cu_seqlens, int num_seqs, int max_seqlen,
                                   int total_tokens, int H, int d, float scale, int causal,
                                   int window, void* stream);
attn_status_t attn_bwd_bf16(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                            float scale, int causal, int window, void* stream);

/*
 * attn_fwd_bf16_varlen -- attn_fwd_bf16 over variable-length sequences packed
 * without padding.
 *
 * [YT] §1.1 从FlashAttention到V3的迭代路径 (support for variable sequence lengths).
 * Sequence s is tokens [cu_seqlens[s], cu_seqlens[s+1]); each sequence attends only
 * within itself, and causal / window masks apply to positions inside it (its first
 * token is position 0).  Per sequence and head the result is attn_fwd_bf16's.
 *   q, k, v : const bf16 [T, H, d] (token-major, then head, then d)
 *   o       : bf16 [T, H, d], written for every token of every sequence
 *   lse     : float [H, T], written likewise (natural log)
 *   cu_seqlens : const int32 [num_seqs + 1] in DEVICE memory, non-decreasing from 0
 *             to total_tokens.  Read on the device only; offsets outside [0, T] are
 *             clamped there, so a bad table gives wrong results, never a stray access.
 *   num_seqs >= 1, H >= 1, total_tokens = T >= 0
 *   max_seqlen : >= the longest sequence and <= T (sizes the work; a longer sequence
 *             would leave rows unwritten); 0 or T == 0: nothing to do, ATTN_OK (the
 *             tensor pointers may then be null)
 *   d in {64, 128, 256}; scale, causal, window as attn_fwd_bf16
 * Alignment: q, k, v, o 16 bytes; lse, cu_seqlens 4 bytes.
 */
attn_status_t attn_fwd_bf16_varlen(const void* q, const void* k, const void* v, void* o,
                                   float* lse, const int* cu_seqlens, int num_seqs,
                                   int max_seqlen, int total_tokens, int H, int d, float scale,
                                   int causal, int window, void* stream);

/*
 * attn_decode_bf16_paged -- one decoding step of attention over a paged KV cache.
 *
 * [JJ] §3 总结 (decoding produces tokens one at a time over a cache of earlier keys
 * and values) and [WGC] 局限性与后续方向 item 2 (PagedAttention KV-cache management).
 * For sequence b with seq_lens[b] = L cached tokens (its nq newest included) and head
 * h, query i is the token at position L - nq + i and attends to keys 0 .. L - nq + i:
 *     O = softmax(scale * q K^T) V over those keys, LSE = natural log of the sum.
 * Key t of sequence b is row t % page_size of page page_table[b][t / page_size].
 *   q          : const bf16 [B, H, nq, d]; 1 <= nq <= 8
 *   k_cache, v_cache : const bf16 [num_pages, H, page_size, d]
 *   page_table : const int32 [B, max_pages] (device); entries are clamped to
 *                [0, num_pages) on the device, so a bad table never reads outside
 *   seq_lens   : const int32 [B] (device); clamped to [0, max_pages * page_size];
 *                rows of a sequence shorter than nq get O = 0, LSE = -inf
 *   o, lse     : bf16 [B, H, nq, d], float [B, H, nq], written
 *   d in {64, 128, 256}; page_size a power of two <= 65536; B * H <= 65535
 *   num_splits : key splits per (sequence, head); 0 picks about sixteen CTAs per SM
 *   workspace  : device memory of attn_decode_workspace_bytes(...) bytes (16-byte
 *                aligned; may be NULL when that is 0).  With num_splits = 0 a smaller
 *                workspace lowers the splits to what fits; with num_splits > 0 it is
 *                ATTN_ERR_INVALID_ARG.
 * HBM-bound: the keys and values of every sequence are read once per call.
 */
size_t attn_decode_workspace_bytes(int B, int H, int nq, int d, int page_size, int max_pages,
                                   int num_splits);
attn_status_t attn_decode_bf16_paged(const void* q, const void* k_cache, const void* v_cache,
                                     const int* page_table, const int* seq_lens, void* o,
                                     float* lse, int B, int H, int nq, int d, int page_size,
                                     int num_pages, int max_pages, float scale, int num_splits,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_bf16_paged_noalloc -- attn_decode_bf16_paged without a caller workspace.
 *
 * The pages have no counterpart to this entry point: it exists for callers that
 * cannot allocate device memory when they decode.  Examples are an inference engine
 * that divided the GPU's memory among its parts at start-up and hands a kernel only
 * the tensors it computes on, and a latency-bound decoding loop in which cudaMalloc
 * would synchronise the device and stall the other streams.  Such a caller passes
 * only its inputs and outputs; the split partials go to a 16 MiB array
 * (4,194,304 floats, a file-scope static device array of the library) that every
 * device which loads the library holds until the process exits.  The entry point
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *   Set-up: the first call of any entry point of this library on a device looks up
 *   that array's device address (cudaGetSymbolAddress, with the device current) and
 *   caches it.  Make that first call before any stream capture begins.
 *   Limit: the partials need B * H * splits * nq * (d + 1) * 4 bytes.  With
 *   num_splits = 0 the plan shrinks to the splits that fit (one split needs no
 *   partials); num_splits > 0 beyond 16 MiB returns ATTN_ERR_INVALID_ARG and
 *   launches nothing.
 *   Sharing: every call uses the same array and leaves its partials there.  Nothing
 *   in it has to start at zero, because every split writes all of its partials
 *   before the merge reads them.  Calls that overlap on the GPU race on the array:
 *   issue calls on one device on one stream, or order the streams yourself.
 *   attn_decode_bf16_paged with a workspace per stream has no such rule.
 */
attn_status_t attn_decode_bf16_paged_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int* page_table,
                                             const int* seq_lens, void* o, float* lse, int B,
                                             int H, int nq, int d, int page_size, int num_pages,
                                             int max_pages, float scale, int num_splits,
                                             void* stream);

/*
 * attn_quantize_fp8_blockwise -- per-block FP8-E4M3 quantisation.
 *
 * [WGC] §3 FP8 量化与精度保持 (per-block dynamic scale onto the FP8 range, whose
 * largest magnitude is 448); [JJ] §1.5 低精度FP8 (E4M3: 4 exponent, 3 mantissa
 * bits) and §1 item 3 (块量化).  For each head and each block of `block`
 * consecutive rows (all d columns):
 *     amax = max |x|,  scale = amax / 448 (IEEE fp32; 1 when amax == 0),
 *     x8   = E4M3(x / scale) with IEEE fp32 division, round-to-nearest-even,
 *            saturating to +-448.
 *   x      : const bf16 [B, H, N, d]
 *   x8     : uint8 (E4M3 codes) [B, H, N, d], written
 *   scales : float [B, H, ceil(N / block)], written; x ~= x8 * scales[block of row]
 *   block  : 128, or 64 (the head-dim-aware block of Q and K at d = 64, see
 *            attn_fp8_qk_block_rows); else ATTN_ERR_UNSUPPORTED.  d % 16 == 0, d <= 256
 */
attn_status_t attn_quantize_fp8_blockwise(const void* x, void* x8, float* scales, int B, int H,
                                          int N, int d, int block, void* stream);

/*
 * attn_quantize_fp8_hadamard -- incoherent processing, then per-block FP8-E4M3
 * quantisation.
 *
 * [JJ] §1 item 3 and its summary (块量化和无相关处理: block quantisation together
 * with incoherent processing, credited with a 2.6x lower FP8 error).  The pages do
 * not spell out the transform; here each row of x is multiplied by the
 * orthonormal Walsh-Hadamard matrix H_d / sqrt(d) (H_d[j][k] = (-1)^popcount(j & k))
 * and the result is quantised exactly as attn_quantize_fp8_blockwise does.  Apply
 * it to Q and K, not V: the rotation is orthogonal, so scores computed from the
 * rotated Q and K equal Q K^T, while an outlier in a row is spread over all d
 * coordinates and the block scale no longer has to cover it alone.
 * The rotated values are computed in fp32: the butterfly sweep h = 1, 2, ..., d/2
 * (each pair i, i + h with (i & h) == 0 becomes a + b, a - b, in that order of
 * stages), then a multiply by fp32(1 / sqrt(d)) (the double 1/sqrt(d) rounded
 * once).  Codes and scales are therefore a pure function of x.
 *   x, x8, scales, block : as attn_quantize_fp8_blockwise
 *   d in {64, 128, 256} (else ATTN_ERR_UNSUPPORTED)
 * The outputs feed attn_fwd_fp8 unchanged (descale_q / descale_k = these scales).
 */
attn_status_t attn_quantize_fp8_hadamard(const void* x, void* x8, float* scales, int B, int H,
                                         int N, int d, int block, void* stream);

/*
 * attn_quantize_fp8_blockwise_fmt -- attn_quantize_fp8_blockwise into either FP8 format.
 *
 * format ATTN_FP8_E4M3: exactly attn_quantize_fp8_blockwise.  format ATTN_FP8_E5M2
 * ([JJ] §1.5 and [WGC] §3 name both formats): scale = amax / 57344 (IEEE fp32; 1 when
 * amax == 0) and x8 = E5M2(x / scale), round-to-nearest-even, saturating to +-57344.
 * format ATTN_FP8_E4M3_POW2 ([WGC] §3 asks only for a per-block scale): E4M3 codes with
 * scale = the smallest power of two >= fp32(amax / 448), so x / scale is exact; used for V
 * it lets attn_fwd_fp8_fmt fold the ratio of two blocks' scales into P exactly.
 * Arguments as attn_quantize_fp8_blockwise; another format is ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_quantize_fp8_blockwise_fmt(const void* x, void* x8, float* scales, int B,
                                              int H, int N, int d, int block, int format,
                                              void* stream);

/*
 * attn_fwd_fp8 -- the forward pass with both matmuls on FP8-E4M3 operands.
 *
 * [WGC] §3 FP8 量化与精度保持 (FP8 inputs, FP32 accumulation, 16-bit output) and
 * [JJ] §2.3 (FP8 tensor-core GEMMs in the forward pass).
 *   q8, k8, v8 : const E4M3 [B, H, N, d] as written by attn_quantize_fp8_blockwise
 *   descale_q/k/v : const float [B, H, N / 128], the matching `scales`
 *                   (x ~= x8 * descale for the 128-row block of the row)
 *   o, lse, scale, causal, window : as attn_fwd_bf16
 *   d in {64, 128, 256}; N % 128 == 0 (else ATTN_ERR_UNSUPPORTED)
 * Scores are descaled per (query block, key block) inside the softmax.  P is
 * rounded to E4M3 as p * 2^8 (p <= 1 against the exact running maximum); the V
 * descale of each key block is applied to the fp32 O accumulator, which is
 * rescaled by alpha * dv(t-1) / dv(t) before P(t) V8(t) is added.
 */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                           const float* descale_q, const float* descale_k,
                           const float* descale_v, void* o, float* lse, int B, int H, int N,
                           int d, float scale, int causal, int window, void* stream);

/*
 * attn_fwd_fp8_fmt -- attn_fwd_fp8 with a choice of formats.
 *
 * Mixed FP8 formats ([JJ] §1.5: E5M2 trades precision for range): q8 and k8 are both
 * qk_format codes (ATTN_FP8_E4M3, ATTN_FP8_E5M2 or ATTN_FP8_E4M3_POW2, from
 * attn_quantize_fp8_blockwise_fmt), v8 is E4M3 (v_format ATTN_FP8_E4M3) or E4M3 with
 * power-of-two block scales (ATTN_FP8_E4M3_POW2), and P is rounded to E4M3 as in
 * attn_fwd_fp8, so each of the two matmuls multiplies two operands of one type.  With
 * power-of-two V scales the kernel applies V's descale through P's exponent and rescales
 * the O accumulator only when a row's max or the largest V scale so far grows, instead
 * of on every key tile; v_format ATTN_FP8_E4M3_POW2 with other scales gives wrong results.
 * qk_format = v_format = ATTN_FP8_E4M3 is exactly attn_fwd_fp8.  Other arguments and
 * errors as attn_fwd_fp8; another format is ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fwd_fp8_fmt(const void* q8, const void* k8, const void* v8,
                               const float* descale_q, const float* descale_k,
                               const float* descale_v, void* o, float* lse, int B, int H, int N,
                               int d, float scale, int causal, int window, int qk_format,
                               int v_format, void* stream);

/*
 * attn_fwd_schedule -- how a batched forward call (attn_fwd_bf16, attn_fwd_fp8 and its
 * variants) with these sizes and mask would spread its work over sm_count SMs: the
 * persistent grid and its walk over the work units ([YT] §1.2 asks for the work to be
 * balanced over the SMs).  A diagnostic: no device memory, stream or kernel is touched.
 *
 * A work unit is (head, query block of 256 rows; 128 at d = 256); sub-unit s is half
 * s & 1 of the complementary pair s >> 1 of query blocks (nq-1-k, k) of a head.
 *   out : int[8], written: [0] walk (0 whole pairs -- causal masks; 1 single units with a
 *         plain stride -- no mask, when that takes fewer rounds; 2 single units in
 *         rotated rounds -- windows), [1] grid (CTAs), [2] sub-units, [3..6] the walk's
 *         constants first, a, m, step: CTA c starts at sub-unit c * first and after s goes
 *         to s + 1 when (s + a) % m == 0, else to s + 1 + step, while s < out[2],
 *         [7] query blocks per head
 *   d in {64, 128, 256} (else ATTN_ERR_UNSUPPORTED); B, H, N, sm_count >= 1 and out
 *   non-null (else ATTN_ERR_INVALID_ARG)
 */
attn_status_t attn_fwd_schedule(int B, int H, int N, int d, int causal, int window,
                                int sm_count, int* out);

/*
 * attn_fp8_qk_block_rows -- rows per Q and K scale block under head-dim-aware
 * scaling: min(d, 128) (0 for d < 1).
 *
 * [WGC] §3 FP8 量化与精度保持 (头维度感知量化): the scaling is tuned separately for
 * head dims 64 and 128 so that small head dims do not lose precision; no rule is
 * given.  Reading: Q and K, whose products run over the d entries of a row, get
 * blocks of min(d, 128) rows -- 64 at d = 64, the 128 rows of the FP8 workload at
 * d >= 128 -- and V keeps 128-row blocks at every d (its error in O averages over
 * keys, not over d).  On the FP8 workload's distribution at d = 64 this lowers the
 * error against unquantised attention; 64-row V blocks change nothing measurable.
 */
int attn_fp8_qk_block_rows(int d);

/*
 * attn_fwd_fp8_blocks -- attn_fwd_fp8_fmt with the height of the Q and K scale blocks
 * as a parameter, for head-dim-aware scaling.
 *   qk_block      : 64 or 128 (else ATTN_ERR_UNSUPPORTED): rows per scale block of Q
 *                   and K; attn_fp8_qk_block_rows(d) gives the head-dim-aware value
 *   descale_q, descale_k : const float [B, H, N / qk_block], the `scales` that
 *                   attn_quantize_fp8_blockwise(_fmt) wrote with block = qk_block
 *   descale_v     : const float [B, H, N / 128] (V is quantised with block = 128)
 * A 128-key tile then spans two K blocks when qk_block = 64; the softmax applies each
 * 64-key half's descale to its own scores.  qk_block = 128 is exactly attn_fwd_fp8_fmt.
 * Other arguments and errors as attn_fwd_fp8_fmt.
 */
attn_status_t attn_fwd_fp8_blocks(const void* q8, const void* k8, const void* v8,
                                  const float* descale_q, const float* descale_k,
                                  const float* descale_v, void* o, float* lse, int B, int H,
                                  int N, int d, float scale, int causal, int window,
                                  int qk_format, int v_format, int qk_block, void* stream);

/* Static English text for a status code (never NULL). */
const char* attn_status_string(attn_status_t status);

/*
 * attn_get_device_status -- synchronise `stream`, then read and clear the status
 * word of the current device: ATTN_OK, or ATTN_ERR_TIMEOUT when a kernel gave up
 * on an internal wait since the last read.  Returns ATTN_ERR_CUDA when the
 * synchronisation itself fails (for instance after a device fault).
 */
attn_status_t attn_get_device_status(void* stream);

/*
 * attn_selftest_wait_timeout -- diagnostic for the failure path every kernel above
 * shares.  Launches one small kernel that waits, with the same bounded mbarrier
 * wait the attention and quantiser kernels use, on a barrier nothing will ever
 * arrive on.  After `timeout_ns` the wait gives up, the kernel records
 * ATTN_ERR_TIMEOUT in the device status word and returns normally, so the
 * context stays usable; read the word with attn_get_device_status().
 *   timeout_ns : 1 .. 2e9 (else ATTN_ERR_INVALID_ARG)
 */
attn_status_t attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/*
 * attn_selftest_fwd_withheld_load, attn_selftest_quant_withheld_load,
 * attn_selftest_bwd_withheld_load -- diagnostics for the abort path of the real
 * kernels (no page describes them: they test this library's failure detection).
 * Each runs the production kernel of attn_fwd_bf16 (scale 1/sqrt(d), no window),
 * of attn_quantize_fp8_blockwise (E4M3, block 128) or of attn_bwd_bf16 on the
 * given tensors, with two differences: every wait is bounded by `timeout_ns`
 * instead of the usual 4 s, and in every CTA the load with index `withheld`
 * (0-based, counted over that CTA's K/V tiles, its 128-row blocks, or its
 * backward ring tiles) is never issued.  The waits on it run out; the CTA raises
 * its abort flag, lets the copies and MMAs it already issued finish, frees its
 * tensor memory and exits, and ATTN_ERR_TIMEOUT is recorded for
 * attn_get_device_status().  The outputs are then unspecified; the context stays
 * usable.  A CTA that never reaches load `withheld` finishes normally.
 * Arguments are as for the production entry points, plus
 *   withheld   : >= 0
 *   timeout_ns : 1 .. 2e9 (else ATTN_ERR_INVALID_ARG)
 */
attn_status_t attn_selftest_fwd_withheld_load(const void* q, const void* k, const void* v,
                                              void* o, float* lse, int B, int H, int N, int d,
                                              int causal, int withheld,
                                              unsigned long long timeout_ns, void* stream);
attn_status_t attn_selftest_quant_withheld_load(const void* x, void* x8, float* scales, int B,
                                                int H, int N, int d, int withheld,
                                                unsigned long long timeout_ns, void* stream);
attn_status_t attn_selftest_bwd_withheld_load(const void* q, const void* k, const void* v,
                                              const void* o, const void* dout, const float* lse,
                                              void* dq, void* dk, void* dv, void* workspace,
                                              size_t workspace_bytes, int B, int H, int N, int d,
                                              int causal, int withheld,
                                              unsigned long long timeout_ns, void* stream);

/*
 * attn_selftest_fp8_convert -- diagnostic: the device's FP8 conversion (the one the
 * quantisers use: round to nearest even, saturating to the format's largest finite
 * value) applied to the fp32 bit patterns first .. first + count - 1, so that a test
 * can compare it with an independent encoder over all 2^32 patterns.  [JJ] §1.5
 * (E4M3 and E5M2).
 *   codes  : uint8 [count] on the device, 16-byte aligned, written: codes[i] is the
 *            code of the float whose bit pattern is first + i
 *   count  : a positive multiple of 8 with first + count <= 2^32
 *   format : ATTN_FP8_E4M3 or ATTN_FP8_E5M2 (else ATTN_ERR_INVALID_ARG)
 */
attn_status_t attn_selftest_fp8_convert(unsigned int first, size_t count, int format,
                                        void* codes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
