/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Exact scaled-dot-product attention O = softmax(s*QK^T)V computed tile by
 * tile with the online-softmax running max / sum so that the N x N score and
 * probability matrices never reach device memory.  Operations:
 *
 *   attn_fwd     fused forward with per-row logsumexp, causal masking and
 *                grouped-query heads (lecture notes "Optimizing Attention for
 *                Modern Hardware: FlashAttention 1-4", sections 2.2 tiling and
 *                rescaling, 2.5 causal block skipping, 2.6 logsumexp, 3.1 loop
 *                order, 3.2 delayed normalisation, 4.5 persistent kernel and
 *                LPT schedule, 5.3 conditional rescaling; "Flash Attention 3/4
 *                notes", FA4 section 1 pipeline and section 3 causal schedule);
 *   attn_fwd_varlen  the same forward over a packed batch of sequences of
 *                different lengths (row offsets per sequence);
 *   attn_fwd_fp8 the forward on E4M3 operands with one scale per 128-row
 *                block, after attn_fp8_quantize (optionally rotating Q and K
 *                by a random-sign Hadamard matrix);
 *   attn_bwd     the gradients dQ, dK, dV from the forward's logsumexp;
 *   attn_decode  single-query decode over a KV cache with split-KV
 *                (Flash-Decoding): each split produces a partial (m, l, o) and
 *                a combine step merges the splits by log-sum-exp (lecture
 *                notes section 6.1 and exercise 3; "FlashAttention tiling &
 *                online softmax" section 7.1), with query heads that share a
 *                KV head packed as rows of one tile (lecture notes 6.2);
 *                attn_decode_paged reads the cache through a block table.
 *
 * Conventions shared by every entry point
 *   - Pointers named q/k/v/o/lse/k_cache/v_cache/seqlens/workspace are DEVICE
 *     pointers.  The caller allocates and owns every buffer it passes,
 *     workspaces included; no entry point allocates device memory.  The
 *     library's own device memory is static tables loaded with it (work
 *     queues, merge counters, the error word, attn_decode_noalloc's scratch).
 *     Tensor data must be 16-byte aligned.
 *   - Per-device state (SM count, the error word's address, the scratch
 *     address) is looked up on the first call on each device and kept for the
 *     life of the process: resetting a device (cudaDeviceReset) after the
 *     library has used it is not supported.
 *   - Tensors are row-major and contiguous: [B, H, N, d] (d fastest) unless
 *     an entry point states another layout (packed batches, paged caches,
 *     transposed FP8 codes).
 *   - bf16 means IEEE-style bfloat16 (1-8-7).  Accumulation is fp32.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Host-side argument checks run before anything is
 *     enqueued; a rejected call enqueues nothing.  Errors are returned, never
 *     printed or thrown.
 *   - Device-side faults of the algorithm itself (a bounded wait that ran
 *     out, an out-of-range sequence length) are recorded in a per-device error
 *     word that attn_last_device_error() reads.
 *   - Head mapping for grouped-query attention: query head hq uses KV head
 *     hq / (Hq / Hkv) (contiguous groups).
 *   - Causal masking is aligned bottom-right: query row i may attend key j iff
 *     j <= i + (Nk - Nq).  With Nq == Nk that is j <= i.
 *   - LSE is the natural-log logsumexp of the scaled scores of a row:
 *     LSE_i = log sum_j exp(scale * q_i . k_j).
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or value   */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement  */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed             */
    ATTN_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out            */
    ATTN_ERR_WORKSPACE = 5     /* workspace missing, too small or misaligned    */
} attn_status_t;

typedef enum {
    ATTN_OUT_BF16 = 0,         /* O written as bf16 (round-to-nearest-even)     */
    ATTN_OUT_F32 = 1           /* O written as fp32                              */
} attn_out_dtype_t;

/*
 * attn_fwd -- fused exact attention forward.
 *
 *   q    bf16 [B, Hq,  Nq, d]        k, v  bf16 [B, Hkv, Nk, d]
 *   o    [B, Hq, Nq, d], element type per o_dtype (bf16 or fp32)
 *   lse  fp32 [B, Hq, Nq] natural-log logsumexp per row, or NULL to skip it
 *   scale  softmax scale (typically 1/sqrt(d)); finite and >= 0
 *   causal 0 or 1 (bottom-right aligned; requires Nq <= Nk)
 *
 * Supported: 8 <= d <= 256 with d % 8 == 0: d <= 128 runs on the 64- or
 *            128-column kernel (two 128-row Q tiles per CTA), 128 < d <= 256
 *            on the 192- or 256-column kernel (one Q tile per CTA, 128-key
 *            K/V tiles, no tail split); other d are padded to the next of
 *            these with the columns past d read as zero and never written.
 *            Hq % Hkv == 0; 1 <= Nq, Nk <= 2^24; B*Hq and B*Hkv <= 2^24.
 *            Other d -> ATTN_ERR_UNSUPPORTED.
 * Numerics: scores and O accumulate in fp32; the probabilities that multiply V
 * are rounded to bf16.  The logsumexp uses the sum of the unrounded
 * probabilities; O is divided by that sum plus, per KV tile, the rounding
 * error of the tile's largest rounded probability.
 * Work distribution: the kernel's CTAs take units from the attn_fwd_schedule
 * list through a device-side queue (one of 256 slots per launch, rotated by
 * the library and left zeroed when the kernel ends), so at most 256 attn_fwd
 * launches may be in flight at the same time.  Tail units may be split along
 * the KV range (attn_fwd_split_plan); their partial results go to the
 * caller's workspace.
 *   workspace  device memory of at least attn_fwd_workspace_size(...) bytes,
 *            16-byte aligned, or NULL when that size is 0; contents need no
 *            initialisation and are garbage afterwards.  Launches that may
 *            overlap on the GPU (different streams) need separate workspaces.
 * Returns ATTN_OK once the kernel is enqueued; ATTN_ERR_WORKSPACE for a
 * missing, short or misaligned workspace (checked after the arguments).
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                       float scale, attn_out_dtype_t o_dtype, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * attn_fwd_workspace_size -- bytes of device workspace attn_fwd needs for
 * this shape on the current device: the partial results of the tail units it
 * splits (per piece and per 32 query rows, (d' + 3) x 32 fp32 values with
 * d' = 64 or 128: O / l, m, l, lx), 0 when it splits none (causal launches,
 * unit counts that fill the SMs' last round, d > 128).  The split depends on
 * the device's SM count, so query on the device that will run the launch.
 * Returns 0 for arguments attn_fwd would reject, or when no device answers.
 */
size_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal);

/*
 * attn_fwd_varlen -- attn_fwd over a packed batch of B sequences of different
 * lengths.  Sequence b is query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and
 * key rows [cu_seqlens_k[b], cu_seqlens_k[b+1]); it attends only to its own
 * keys (causal: bottom-right aligned within the sequence).
 *
 *   q    bf16 [total_q, Hq,  d]      k, v  bf16 [total_k, Hkv, d]
 *   o    [total_q, Hq, d], element type per o_dtype
 *   lse  fp32 [Hq, total_q], or NULL
 *   cu_seqlens_q, cu_seqlens_k  DEVICE int32 [B + 1], non-decreasing, from 0
 *        or more up to total_q / total_k (rows outside every sequence are
 *        neither read nor written)
 *   max_seqlen_q, max_seqlen_k  upper bounds of the lengths (host ints)
 *
 * Supported as attn_fwd (8 <= d <= 256, d % 8 == 0; d > 128 on the 192- or
 * 256-column kernel); 1 <= total_q,
 * total_k <= 2^30; max lengths in [1, 2^24].  The lengths live on the device, so their checks run there: a
 * sequence whose offsets leave [0, total], decrease, exceed the maximum
 * length, give query rows without keys, or (causal) more queries than keys
 * is not computed (its O and LSE rows are left as they were) and
 * attn_last_device_error() then reports ATTN_ERR_INVALID_ARG.  A sequence of
 * length 0 is skipped.  Numerics as attn_fwd; no KV tail split.  Loads stop
 * at each sequence's last row (no value of another sequence, NaN included,
 * reaches a result).  Uses a work-queue slot as attn_fwd.
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int total_q, int total_k, int max_seqlen_q,
                              int max_seqlen_k, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, void* stream);

/*
 * attn_fp8_quantize -- block quantization to E4M3 (lecture notes "Optimizing
 * Attention for Modern Hardware: FlashAttention 1-4", 4.4; "Flash Attention
 * 3/4 notes", FA3 section 2: one scale per block, incoherent processing).
 *
 *   x        bf16 [B, H, N, d] (device)
 *   signs    NULL, or d int8 values +-1 (device): each row x is first replaced
 *            by H (s o x), H the unnormalised Sylvester-Hadamard matrix
 *            (entries +-1), computed in fp32 by the fast Walsh-Hadamard
 *            transform (stages h = 1, 2, ..., d/2; pairs (i, i+h) become
 *            (a+b, a-b)).  Rotating Q and K with the same signs multiplies
 *            their scores by d (pass rotated = 1 to attn_fwd_fp8).
 *   codes    E4M3 codes (device), [B, H, N, d] when transpose = 0, or
 *            [B, H, d, Np] with Np = ceil(N/16)*16 when transpose = 1 (the
 *            layout attn_fwd_fp8 wants for V; the padding keys hold 0);
 *            attn_fp8_codes_bytes() bytes
 *   descale  fp32 [B, H, ceil(N/128)]: for each block of 128 rows,
 *            amax / 448 with amax the block's largest |value| (1 for an
 *            all-zero block); codes are E4M3(fp32(x * (448 / amax))) rounded to
 *            nearest even, so code * descale approximates x.
 * Supported: d = 128; B*H <= 65535.  Asynchronous on `stream`.
 */
size_t attn_fp8_codes_bytes(int B, int H, int N, int d, int transpose);
size_t attn_fp8_descale_count(int B, int H, int N);
attn_status_t attn_fp8_quantize(const void* x, void* codes, float* descale, const int8_t* signs,
                                int B, int H, int N, int d, int transpose, void* stream);

/*
 * attn_fwd_fp8 -- attn_fwd on E4M3 operands from attn_fp8_quantize:
 *
 *   q8  [B, Hq, Nq, 128] codes, q_descale [B, Hq, ceil(Nq/128)]
 *   k8  [B, Hkv, Nk, 128] codes, k_descale [B, Hkv, ceil(Nk/128)]
 *   vt8 [B, Hkv, 128, Np] transposed codes, v_descale [B, Hkv, ceil(Nk/128)]
 *   o, lse, causal, o_dtype as attn_fwd; scale as attn_fwd: the softmax
 *   scale of the original (unrotated) problem
 *   rotated  1 when q8 and k8 were made by attn_fp8_quantize with the same
 *            signs (rotated Q and K): their scores are then d times the
 *            original ones and the library applies scale / d; 0 otherwise.
 *
 * Computes softmax(scale * Q^ K^^T) V^ over the dequantized operands (code *
 * block descale) with fp32 accumulation; the probabilities are rounded to
 * E4M3 before the P.V product (in a frame that carries V's block scale and a
 * factor 2^4, so they stay within E4M3's range), and the row sums follow the
 * unrounded ones as in attn_fwd.  LSE is the natural-log logsumexp of the
 * scaled scores.  Supported: d = 128, other limits as attn_fwd.  Uses one of
 * 256 queue slots per launch, as attn_fwd.
 */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                           const float* k_descale, const float* v_descale, void* o, float* lse,
                           int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                           int rotated, attn_out_dtype_t o_dtype, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs: two
 * fp32 row vectors (D and the logsumexp in base 2) over query rows padded to
 * whole 128-row tiles (8 * B*Hq*ceil(Nq/128)*128 bytes).  Returns 0 for
 * shapes attn_bwd would reject.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/*
 * attn_bwd -- gradients of attn_fwd (lecture notes "Optimizing Attention for
 * Modern Hardware: FlashAttention 1-4", 2.6: P recomputed from the stored
 * logsumexp, D = rowsum(dO o O), dS = P o (dP - D)):
 *
 *   dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO
 *
 * with dK and dV summed over each KV head's query-head group (GQA).
 *
 *   q, dout  bf16 [B, Hq, Nq, d]       k, v  bf16 [B, Hkv, Nk, d]
 *   o        the forward's output [B, Hq, Nq, d], element type per o_dtype
 *   lse      fp32 [B, Hq, Nq], the forward's natural-log logsumexp
 *   dq       [B, Hq, Nq, d];  dk, dv  [B, Hkv, Nk, d]; element type per
 *            grad_dtype (bf16 round-to-nearest-even, or fp32)
 *   causal, scale  as passed to attn_fwd
 *   workspace  device memory of at least attn_bwd_workspace_size bytes,
 *            16-byte aligned; contents need no initialisation; not used after
 *            the call's kernels finish.
 *
 * Supported: 8 <= d <= 256 with d % 8 == 0 (attn_fwd's limits otherwise:
 * Hq % Hkv == 0, causal needs Nq <= Nk).  d <= 128 runs on the kernels
 * described below; 128 < d <= 256 on kernels built for 256 columns with other
 * tile shapes (the dK/dV pass per 128 keys and per 128-column half of d over
 * 64-row Q tiles, the dQ pass per 128 query rows over 64-key tiles, one CTA
 * per item).  Pointers 16-byte aligned (lse 4-byte).  The caller owns every
 * buffer.  Three kernels run in order on `stream`: a per-row pass (D, the LSE
 * in base 2), a K/V-outer pass (an item per (b, KV head, 128-key tile): dK
 * and dV accumulated in tensor memory over the group's query heads and Q
 * tiles, written once) and a Q-outer pass (an item per (b, query head,
 * 128-row Q tile): dQ accumulated in tensor memory over the K/V tiles,
 * written once); for d <= 128 both passes run at most one CTA per SM, each
 * CTA taking every (grid size)-th item.  No atomics: every gradient is bit-identical from run to
 * run.  S and dP are computed in both passes (lecture notes exercise 6).
 * Numerics: scores and all products accumulate in fp32; P and dS are rounded
 * to bf16 before the P.dO, dS.Q and dS.K products.  Returns ATTN_OK once the kernels are enqueued;
 * ATTN_ERR_WORKSPACE for a missing or short workspace.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                       attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * attn_bwd_varlen_workspace_size -- bytes of device workspace attn_bwd_varlen
 * needs: D and the base-2 logsumexp for every query head over each
 * sequence's rows padded to whole 128-row tiles (8 * Hq * (total_q + 132 B)
 * bytes, rounded up).  Returns 0 for arguments attn_bwd_varlen would reject.
 */
size_t attn_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int d);

/*
 * attn_bwd_varlen -- gradients of attn_fwd_varlen: attn_bwd's computation for
 * every sequence of a packed batch (each sequence an independent problem,
 * bottom-right causal alignment per sequence).
 *
 *   q, dout  bf16 [total_q, Hq, d]      k, v  bf16 [total_k, Hkv, d]
 *   o        attn_fwd_varlen's output [total_q, Hq, d], element type per o_dtype
 *   lse      fp32 [Hq, total_q], attn_fwd_varlen's logsumexp
 *   dq       [total_q, Hq, d];  dk, dv  [total_k, Hkv, d]; element type per
 *            grad_dtype
 *   cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k  as attn_fwd_varlen
 *   workspace  device memory of at least attn_bwd_varlen_workspace_size bytes,
 *            16-byte aligned; contents need no initialisation.
 *
 * Supported: 8 <= d <= 256 (d % 8 == 0); the other limits of attn_fwd_varlen.
 * The same three kernels as attn_bwd (D and the base-2 LSE per row, the
 * K/V-outer pass, the Q-outer pass; for 128 < d <= 256 the 256-column passes)
 * read the packed rows through the packed forward's ragged tensor maps; CTAs
 * cover every sequence at the longest lengths, and the tiles past a
 * sequence's end have no work.  A sequence whose
 * offsets fail the checks of attn_fwd_varlen is not computed (its gradient
 * rows are left as they were) and attn_last_device_error() then reports
 * ATTN_ERR_INVALID_ARG.  Rows outside every sequence are neither read nor
 * written.  Gradients are bit-identical from run to run.  Returns ATTN_OK once
 * the kernels are enqueued; ATTN_ERR_WORKSPACE for a missing or short
 * workspace; ATTN_ERR_UNSUPPORTED for d outside the supported range.
 */
attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int total_q, int total_k, int max_seqlen_q,
                              int max_seqlen_k, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode needs
 * for this shape and split request (num_splits as passed to attn_decode).
 * Returns 0 for arguments attn_decode would reject.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nmax, int d, int num_splits);

/*
 * attn_decode_paged -- attn_decode over a paged KV cache (the block-table
 * layout decode servers use; lecture notes 6.1 split-KV as in attn_decode).
 *
 *   k_pages, v_pages  bf16 [num_blocks, page_size, Hkv, d]: pages of page_size
 *            consecutive keys, all KV heads of a key together
 *   block_table  int32 [B, max_blocks] (device): logical block i of sequence
 *            b (keys [i*page_size, (i+1)*page_size)) is page block_table[b, i]
 *   seqlens  int32 [B] (device), as for attn_decode, with Nmax = max_blocks *
 *            page_size; only the blocks that hold keys < seqlens[b] are read
 *   page_size a multiple of 64 (ATTN_ERR_UNSUPPORTED otherwise)
 *   workspace  at least attn_decode_workspace_size(B, Hq, Hkv, max_blocks *
 *            page_size, d, num_splits) bytes
 *
 * Everything else (q, o, lse, scale, num_splits, splits and merge, errors) is
 * as for attn_decode, and for the same keys the result is bit-identical to
 * attn_decode on the same values stored contiguously.  A block-table entry
 * outside [0, num_blocks) reads as zeros (it never faults).
 */
attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seqlens, void* o, float* lse,
                                int B, int Hq, int Hkv, long long num_blocks, int page_size,
                                int max_blocks, int d, float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, attn_out_dtype_t o_dtype, void* stream);

/*
 * Number of kernels attn_decode launches for this shape and split request:
 * 1 when the split kernel merges the splits itself (the last split of each
 * (sequence, KV head) to finish merges them; at most 4096 such groups and
 * G * ceil(Nmax / chunk) + 32 floats of merge scratch), else 2 (a combine
 * kernel merges).  Returns -1 for arguments attn_decode would reject.
 */
int attn_decode_kernel_launches(int B, int Hq, int Hkv, int Nmax, int d, int num_splits);

/*
 * attn_decode -- one query token per sequence against a KV cache (split-KV).
 *
 *   q        bf16 [B, Hq, 1, d]
 *   k_cache  bf16 [B, Hkv, Nmax, d]     v_cache  bf16 [B, Hkv, Nmax, d]
 *   seqlens  int32 [B] (device): valid prefix length of each sequence, in
 *            [1, Nmax].  Keys at positions >= seqlens[b] are never read into
 *            the result (they may hold anything, including NaN).  A length
 *            outside [1, Nmax] is clamped into [0, Nmax] and recorded in the
 *            device error word (attn_last_device_error -> INVALID_ARG); a
 *            clamped length of 0 yields O = 0, LSE = -inf.
 *   o        [B, Hq, 1, d] per o_dtype;  lse  fp32 [B, Hq, 1] or NULL
 *   num_splits  0 = choose automatically; k > 0 = cut each sequence's KV
 *            range into chunks of ceil(Nmax / k) keys (rounded up to a multiple
 *            of 64), so a sequence of length Nmax gets (at most) k splits.
 *   workspace   device scratch of at least attn_decode_workspace_size(...)
 *            bytes, 16-byte aligned; contents need no initialisation and are
 *            garbage afterwards.  Concurrent calls must not share it.
 *
 * Supported: 8 <= d <= 256 with d % 8 == 0 (d <= 128 on the 64- or
 * 128-column kernel, 128 < d <= 256 on the 256-column one; the columns past d
 * are read as zero and never written); Hq % Hkv == 0; Hq / Hkv <= 16;
 * 1 <= Nmax <= 2^24.
 */
attn_status_t attn_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nmax, int d, float scale, int num_splits, void* workspace,
                          size_t workspace_bytes, attn_out_dtype_t o_dtype, void* stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart: it is an addition for callers that
 * must not call cudaMalloc, such as a plugin inside a host framework that owns
 * all device memory through its own pool, or a latency-critical loop that
 * cannot afford an allocation's implicit device synchronisation.
 *
 * Same arguments and results as attn_decode, minus the workspace: the split
 * partials go to a scratch array of 16 MiB that the library reserves in
 * device global memory on every GPU that loads it, held until the process
 * exits.  Requests whose attn_decode_workspace_size() exceeds 16 MiB return
 * ATTN_ERR_WORKSPACE without enqueuing anything (use attn_decode with your own
 * workspace for those).  No call allocates device memory.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Nothing in it needs to start at zero: each call writes every
 *     partial before reading it.  Calls that overlap on the GPU (different
 *     streams, or different host threads without ordering) race on it; calls
 *     ordered on one stream do not.
 */
attn_status_t attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int* seqlens, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Nmax, int d, float scale, int num_splits,
                                  attn_out_dtype_t o_dtype, void* stream);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status_t status);

/*
 * attn_last_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a kernel's
 * bounded wait ran out; its outputs are undefined), ATTN_ERR_INVALID_ARG (a
 * decode sequence length was out of range) or ATTN_ERR_CUDA.
 */
attn_status_t attn_last_device_error(void* stream);

/* ---------------------------------------------------------------------------
 * Host-side scheduling logic, exported so it can be inspected and tested.
 * These functions touch no GPU.
 * ------------------------------------------------------------------------- */

/*
 * Split-count rule for uniform-length decode (lecture notes 6.1, exercise 11):
 * over s = 1..max_splits, wave efficiency e(s) = w/ceil(w) with
 * w = units*s/num_sms; return the smallest s with e(s) >= 0.85 * max_s e(s).
 * units = batch x KV heads.  Returns 0 on a bad argument.
 */
int attn_decode_num_splits(int units, int num_sms, int max_splits);

/*
 * Greedy list scheduling (lecture notes 4.5): jobs are taken in the given
 * order (lpt = 0) or longest-first (lpt = 1, stable), each to the currently
 * least-loaded worker, lowest index on ties.  Writes per-worker loads to
 * loads_out[workers] (may be NULL) and returns the makespan (max load), or
 * -1 on a bad argument.
 */
long long attn_list_schedule(const int* costs, int n, int workers, int lpt, long long* loads_out);

/*
 * Number of 128-key KV tiles a block of query rows [row0, row0 + rows) must
 * visit (causal block skipping, lecture notes 2.5): all ceil(Nk / block) tiles
 * without causal masking, else the tiles up to the one holding key
 * row0 + rows - 1 + (Nk - Nq).  `block` is the key-tile height.
 */
int attn_kv_tiles(int row0, int rows, int Nq, int Nk, int causal, int block);

/*
 * Number of work units attn_fwd launches for a shape (a unit = one batch,
 * one query head, one block of 256 query rows = two 128-row Q tiles).
 */
long long attn_fwd_num_units(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal);

/*
 * The order in which attn_fwd's persistent kernel takes its units on a GPU
 * with num_sms SMs: fills units_out[3*i + {0,1,2}] = (b, hq, m_block) for
 * i < n (n must equal attn_fwd_num_units) and, if cost_out is non-NULL,
 * cost_out[i] = the number of (Q tile, KV tile) pairs unit i computes.  Heads
 * are grouped into sections of K/V, sections run in order, and within a
 * section the m-blocks run longest-first (lecture notes 4.5; "Flash Attention
 * 3/4 notes" FA4 section 3).  Non-causal sections span 16 MiB of K/V.  A
 * causal launch takes, of the widths 8, 16, 32, 64 and 128 MiB, the narrowest
 * whose makespan under greedy list scheduling on num_sms workers (each unit
 * costing its KV steps plus 2 for its fixed cost) is within 1 % of the best;
 * num_sms = 0 gives the fixed width of 64 MiB.  Each CTA takes the next unit
 * of this list when it is ready for one (greedy list scheduling, as
 * attn_list_schedule models it).  Returns 0, or -1 on a bad argument.
 */
int attn_fwd_schedule(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms,
                      long long n, int* units_out, int* cost_out);

/*
 * The tail split attn_fwd applies on a GPU with `num_sms` SMs.  Without
 * causal masking all units cost the same; when their count is not a multiple
 * of num_sms, the last units % num_sms units of the schedule (the "tail") are
 * each cut along the KV range into `parts` pieces of near-equal tile counts
 * (piece p of n tiles: tiles [p*n/parts, (p+1)*n/parts)), parts =
 * min(num_sms / tail, KV tiles per unit, 8), so that all pieces run in one
 * round on CTAs that would otherwise idle.  The persistent grid is
 * min(n_full + n_split * parts, num_sms) CTAs.  Each piece keeps its own running max and sums;
 * the last piece of a tail unit to finish merges them by the logsumexp
 * rescaling (lecture notes 6.1 split-KV, 2.2 rescaling).  No split (n_split =
 * 0, parts = 1) for causal launches, when units is a multiple of the grid,
 * when parts < 2 or when the tail exceeds 255 units.  Writes the number of
 * whole units, of split units and the pieces per split unit; returns 0, or -1
 * on a bad argument.
 */
int attn_fwd_split_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms,
                        int* n_full, int* n_split, int* parts);

/*
 * attn_selftest_bounded_wait -- diagnostic of the kernels' bounded waits (every
 * spin in the library's kernels gives up after 2 s, records ATTN_ERR_TIMEOUT in
 * the device error word, and lets the context carry on).  One CTA waits, with
 * the kernels' own wait, on an mbarrier that nothing ever arrives on:
 *   mode 0  the wait runs out (about 2 s); attn_last_device_error() then
 *           reports ATTN_ERR_TIMEOUT;
 *   mode 1  another warp raises the CTA's abort flag after about 1 ms and the
 *           wait returns at once (no error recorded).
 *   result  DEVICE int: 1 = left through the abort flag, 2 = ran out of time,
 *           3 = the phase completed (never expected).
 * Asynchronous on `stream`.
 */
attn_status_t attn_selftest_bounded_wait(int mode, int* result, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
