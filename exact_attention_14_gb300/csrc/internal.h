// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"

namespace gb300 {

// Head dims d in [8, 128], multiples of 8, run on the kernels built for 64 or
// 128 columns: TMA fills the columns past d with zeros on load (they add
// nothing to Q K^T and give zero O columns), and stores skip them.
inline int pad_head_dim(int d) { return d <= 64 ? 64 : 128; }
inline bool head_dim_supported(int d) { return d >= 8 && d <= 128 && d % 8 == 0; }
// The dense forward also takes 128 < d <= 256 (multiples of 8) on the kernels
// built for 192 and 256 columns (one Q tile per CTA; attn_fwd_wide_sm103.cu).
inline bool fwd_head_dim_supported(int d) { return d >= 8 && d <= 256 && d % 8 == 0; }
// Decode takes the same range: d <= 128 on the 64- or 128-column kernel,
// 128 < d <= 256 on the 256-column one.
inline int decode_pad_head_dim(int d) { return d <= 64 ? 64 : (d <= 128 ? 128 : 256); }
inline bool decode_head_dim_supported(int d) { return fwd_head_dim_supported(d); }

struct DeviceInfo {
    int device;
    int num_sms;
    unsigned int* err_word;  // device address of the library's error word
};

// Per-device facts for the current device, initialised once per device.
attn_status_t current_device_info(DeviceInfo* out);

// 3-D bf16 tensor map over a [heads, rows, d] array with a 128-byte-swizzled
// box of (64 elements of d) x box_rows x 1.  Out-of-range rows read as zero.
attn_status_t encode_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int rows,
                                  long long heads, int box_rows);

// 3-D tensor map over an output [heads, rows, d] array (bf16 or fp32), no
// swizzle, box of box_cols x box_rows x 1, for TMA stores of staged tiles.
attn_status_t encode_tmap_out_3d(CUtensorMap* map, void* base, bool f32, int d, int rows,
                                 long long heads, int box_cols, int box_rows);

// 3-D fp32 tensor map over [heads, rows, d] with a 128-byte-swizzled box of
// 32 columns x box_rows x 1 (TMA reduce-add of staged fp32 tiles).
attn_status_t encode_tmap_f32_sw128_3d(CUtensorMap* map, void* base, int d, int rows,
                                       long long heads, int box_rows);

// 4-D bf16 tensor map over a paged KV cache [num_blocks, page_size, Hkv, d]
// with a 128-byte-swizzled box of 64 (d) x 1 (head) x 64 (keys) x 1 (block).
attn_status_t encode_tmap_paged_kv(CUtensorMap* map, const void* base, int d, int Hkv,
                                   int page_size, long long num_blocks);

// 5-D tensor map over a packed [total, heads, d] array (bf16, or fp32 for
// outputs) addressed per sequence: see the ragged layout in fwd_sched.h.  Box of
// box_cols x 1 head x box_rows rows; 128-byte swizzle for the operand loads,
// none for the staged output stores.
attn_status_t encode_tmap_ragged(CUtensorMap* map, const void* base, bool f32, int d, int heads,
                                 int box_cols, int box_rows, bool swizzle128);

// 3-D uint8 tensor map over [heads, rows, inner] with a row pitch in bytes
// (a multiple of 16), 128-byte-swizzled box of box_inner x box_rows x 1.
attn_status_t encode_tmap_u8_3d(CUtensorMap* map, const void* base, int inner, long long pitch,
                                int rows, long long heads, int box_inner, int box_rows);

// FP8: block quantization of bf16 [BH, N, 128] (optionally rotated by the
// sign-flipped Hadamard transform; transposed to [BH, 128, Np] on request), and
// the forward on E4M3 operands (d = 128).
attn_status_t launch_fp8_quantize(const void* x, void* out, float* descale, const int8_t* signs,
                                  int BH, int N, int transpose, cudaStream_t stream,
                                  const DeviceInfo& dev);
attn_status_t launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                             const float* k_descale, const float* v_descale, void* o, float* lse,
                             int B, int Hq, int Hkv, int Nq, int Nk, int causal, float scale,
                             attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev);

// Dense forward.  Bytes of workspace it needs for the partial results of the
// units its tail split cuts into pieces (0 when nothing is split) on a GPU
// with num_sms SMs; launch_fwd takes a workspace of at least that size.
size_t fwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms);
attn_status_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                         attn_out_dtype_t o_dtype, void* workspace, cudaStream_t stream,
                         const DeviceInfo& dev);

// Dense forward for 128 < d <= 256.
attn_status_t launch_fwd_wide(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev);

// Packed variable-length forward: q/o [total_q, Hq, d], k/v [total_k, Hkv, d],
// lse [Hq, total_q]; cu_q / cu_k device int32 [B + 1].
attn_status_t launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                const int* cu_q, const int* cu_k, int B, int Hq, int Hkv,
                                int total_q, int total_k, int max_q, int max_k, int d, int causal,
                                float scale, attn_out_dtype_t o_dtype, cudaStream_t stream,
                                const DeviceInfo& dev);
// The same for 128 < d <= 256.
attn_status_t launch_fwd_wide_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const int* cu_q, const int* cu_k, int B, int Hq, int Hkv,
                                     int total_q, int total_k, int max_q, int max_k, int d,
                                     int causal, float scale, attn_out_dtype_t o_dtype,
                                     cudaStream_t stream, const DeviceInfo& dev);

// Backward: workspace bytes (fp32 dQ accumulator, lse2, D; padded rows).
size_t bwd_workspace_bytes(int B, int Hq, int Nq, int d);
// Packed backward (d <= 128): workspace bytes, and the launch.
size_t bwd_varlen_workspace_bytes(int B, int Hq, int total_q);
attn_status_t launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                const int* cu_q, const int* cu_k, int B, int Hq, int Hkv, int total_q,
                                int total_k, int max_q, int max_k, int d, int causal, float scale,
                                attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype,
                                void* workspace, cudaStream_t stream, const DeviceInfo& dev);
attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                         attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype, void* workspace,
                         cudaStream_t stream, const DeviceInfo& dev);

// Decode: the argument checks of attn_decode (pointers, alignment, shape,
// scale, split request, output type); touches no device.
attn_status_t check_decode_call(const void* q, const void* k_cache, const void* v_cache,
                                const int* seqlens, const void* o, const float* lse, int B, int Hq,
                                int Hkv, int Nmax, int d, float scale, int num_splits,
                                attn_out_dtype_t o_dtype);
// Decode: chunk size in keys for a request (multiple of 64).
int decode_chunk(int Nmax, int B, int Hkv, int num_sms, int num_splits);
size_t decode_workspace_bytes(int B, int Hq, int Nmax, int d, int chunk);
// Decode: whether the split kernel merges the splits itself (else a second
// kernel does); max_splits = ceil(Nmax / chunk).
bool decode_merges_in_kernel(int B, int Hkv, int G, int max_splits, int d);

attn_status_t launch_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                            int Nmax, int d, float scale, int chunk, void* workspace,
                            attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev);
// Paged cache: k/v pages [num_blocks, page_size, Hkv, d], block_table
// [B, max_blocks] (page of logical block i of sequence b); Nmax = max_blocks *
// page_size, page_size a multiple of 64.
attn_status_t launch_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                  const int* block_table, const int* seqlens, void* o, float* lse,
                                  int B, int Hq, int Hkv, long long num_blocks, int page_size,
                                  int max_blocks, int d, float scale, int chunk, void* workspace,
                                  attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace gb300
