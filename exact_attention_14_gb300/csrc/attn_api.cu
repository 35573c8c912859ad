// attn_api.cu -- the C ABI: argument checks, per-device state, tensor-map
// encoding, dispatch to the kernels, status reporting, and the host-side
// scheduling exports declared in attn.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "internal.h"
#include "ptx.cuh"
#include "fwd_sched.h"

namespace gb300 {

// The library's device error word (one per device/context).  Kernels OR
// error bits into it; attn_last_device_error() reads and clears it.
__device__ unsigned int g_attn_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kMaxLen = 1ll << 24;
constexpr long long kMaxHeads = 1ll << 24;
constexpr int kMaxPackedRows = 1 << 30;  // rows of a packed batch (ragged maps, fwd_sched.h)

struct DevState {
    bool ready;
    int num_sms;
    unsigned int* err_word;
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

attn_status_t current_device_info(DeviceInfo* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DevState& s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;  // built for sm_103a only
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_error_word) != cudaSuccess) return ATTN_ERR_CUDA;
        s.num_sms = sms;
        s.err_word = static_cast<unsigned int*>(p);
        s.ready = true;
    }
    out->device = dev;
    out->num_sms = s.num_sms;
    out->err_word = s.err_word;
    return ATTN_OK;
}

static bool load_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return true;
}

attn_status_t encode_tmap_out_3d(CUtensorMap* map, void* base, bool f32, int d, int rows,
                                 long long heads, int box_cols, int box_rows) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * es, (cuuint64_t)d * es * (cuuint64_t)rows};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1u};
    cuuint32_t elem[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          3, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t encode_tmap_paged_kv(CUtensorMap* map, const void* base, int d, int Hkv,
                                   int page_size, long long num_blocks) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)page_size, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2,
                             (cuuint64_t)page_size * Hkv * d * 2};
    cuuint32_t box[4] = {64u, 1u, 64u, 1u};
    cuuint32_t elem[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t encode_tmap_f32_sw128_3d(CUtensorMap* map, void* base, int d, int rows,
                                       long long heads, int box_rows) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)d * 4 * (cuuint64_t)rows};
    cuuint32_t box[3] = {32u, (cuuint32_t)box_rows, 1u};
    cuuint32_t elem[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t encode_tmap_ragged(CUtensorMap* map, const void* base, bool f32, int d, int heads,
                                 int box_cols, int box_rows, bool swizzle128) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    const cuuint64_t es = f32 ? 4 : 2;
    const cuuint64_t rs = (cuuint64_t)heads * d * es;  // row stride (bytes)
    if (rs >= (1ull << 34)) return ATTN_ERR_UNSUPPORTED;
    cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)kRaggedWindow,
                          (cuuint64_t)kRaggedOuterExtent, (cuuint64_t)kRaggedOuterExtent};
    cuuint64_t strides[4] = {(cuuint64_t)d * es, rs, rs, (1ull << 34) - rs};
    cuuint32_t box[5] = {(cuuint32_t)box_cols, 1u, (cuuint32_t)box_rows, 1u, 1u};
    cuuint32_t elem[5] = {1u, 1u, 1u, 1u, 1u};
    CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          5, const_cast<void*>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t encode_tmap_u8_3d(CUtensorMap* map, const void* base, int inner, long long pitch,
                                int rows, long long heads, int box_inner, int box_rows) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)pitch, (cuuint64_t)pitch * (cuuint64_t)rows};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1u};
    cuuint32_t elem[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t encode_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int rows,
                                  long long heads, int box_rows) {
    if (!load_encoder()) return ATTN_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    cuuint32_t elem[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                          strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Diagnostic of the kernels' bounded waits: warp 0 waits, with the same
// mbar_wait every kernel uses, on an mbarrier that nothing ever arrives on.
// mode 0: the wait runs out its time limit; the kernel then ORs kErrTimeout
// into the error word as the real kernels do.  mode 1: warp 1 raises the CTA's
// abort flag after about a millisecond and the wait must return early.
// result: 1 = left through the abort flag, 2 = ran out of time, 3 = the phase
// completed (impossible).
__global__ void attn_selftest_wait_kernel(int mode, int* result, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        const uint64_t t0 = global_timer_ns();
        const bool ok = mbar_wait(smem_u32(&bar), 0, (const volatile int*)&abort_flag);
        const uint64_t waited = global_timer_ns() - t0;
        if (threadIdx.x == 0) {
            if (ok) {
                *result = 3;
            } else if (waited > kWaitLimitNs) {
                *result = 2;
                atomicOr(err, kErrTimeout);
            } else {
                *result = 1;
            }
        }
    } else if (warp == 1 && mode == 1 && threadIdx.x == 32) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
        *((volatile int*)&abort_flag) = 1;
    }
}

}  // namespace gb300

using namespace gb300;

namespace {

attn_status_t check_common(int B, int Hq, int Hkv, int d, float scale, attn_out_dtype_t o_dtype) {
    if (B < 1 || Hq < 1 || Hkv < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * Hq > kMaxHeads || (long long)B * Hkv > kMaxHeads) return ATTN_ERR_INVALID_ARG;
    if (!(scale >= 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (o_dtype != ATTN_OUT_BF16 && o_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

attn_status_t check_fwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        int causal, float scale, attn_out_dtype_t o_dtype) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (lse && !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_common(B, Hq, Hkv, d, scale, o_dtype);
    if (st != ATTN_OK) return st;
    if (Nq < 1 || Nk < 1 || Nq > kMaxLen || Nk > kMaxLen) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return ATTN_ERR_INVALID_ARG;
    if (!fwd_head_dim_supported(d)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

attn_status_t check_decode_shape(int B, int Hq, int Hkv, int Nmax, int d, int num_splits) {
    if (B < 1 || Hq < 1 || Hkv < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * Hq > kMaxHeads || (long long)B * Hkv > kMaxHeads) return ATTN_ERR_INVALID_ARG;
    if (Nmax < 1 || Nmax > kMaxLen) return ATTN_ERR_INVALID_ARG;
    if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
    if (!decode_head_dim_supported(d)) return ATTN_ERR_UNSUPPORTED;
    if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

}  // namespace

// Pointer, shape and value checks of a contiguous-cache decode call (no device
// is touched), shared by attn_decode and attn_decode_noalloc.
attn_status_t gb300::check_decode_call(const void* q, const void* k_cache, const void* v_cache,
                                       const int* seqlens, const void* o, const float* lse, int B,
                                       int Hq, int Hkv, int Nmax, int d, float scale,
                                       int num_splits, attn_out_dtype_t o_dtype) {
    if (!q || !k_cache || !v_cache || !seqlens || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        !aligned4(seqlens))
        return ATTN_ERR_INVALID_ARG;
    if (lse && !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_common(B, Hq, Hkv, d, scale, o_dtype);
    if (st != ATTN_OK) return st;
    return check_decode_shape(B, Hq, Hkv, Nmax, d, num_splits);
}

namespace {

// SM count of the current device, for the size queries (the launches read the
// same per-device value).  -1 when no device can be queried.
int current_num_sms(int* sms) {
    DeviceInfo dev;
    if (current_device_info(&dev) == ATTN_OK) {
        *sms = dev.num_sms;
        return 0;
    }
    return -1;
}

}  // namespace

extern "C" {

size_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal) {
    if (check_common(B, Hq, Hkv, d, 1.0f, ATTN_OUT_BF16) != ATTN_OK) return 0;
    if (Nq < 1 || Nk < 1 || Nq > kMaxLen || Nk > kMaxLen) return 0;
    if ((causal != 0 && causal != 1) || (causal && Nq > Nk)) return 0;
    if (!fwd_head_dim_supported(d)) return 0;
    int sms = 0;
    if (current_num_sms(&sms) != 0) return 0;
    return fwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, causal, sms);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                       attn_out_dtype_t o_dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
    attn_status_t st = check_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, o_dtype);
    if (st != ATTN_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    const size_t need = fwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, causal, dev.num_sms);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return ATTN_ERR_WORKSPACE;
    return launch_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, o_dtype, workspace,
                      static_cast<cudaStream_t>(stream), dev);
}

size_t attn_fp8_codes_bytes(int B, int H, int N, int d, int transpose) {
    if (B < 1 || H < 1 || N < 1 || d != 128 || (transpose != 0 && transpose != 1)) return 0;
    if ((long long)B * H > kMaxHeads || N > kMaxLen) return 0;
    const long long n = transpose ? (long long)(N + 15) / 16 * 16 : (long long)N;
    return (size_t)((long long)B * H * n * d);
}

size_t attn_fp8_descale_count(int B, int H, int N) {
    if (B < 1 || H < 1 || N < 1 || (long long)B * H > kMaxHeads || N > kMaxLen) return 0;
    return (size_t)((long long)B * H * ((N + 127) / 128));
}

attn_status_t attn_fp8_quantize(const void* x, void* codes, float* descale, const int8_t* signs,
                                int B, int H, int N, int d, int transpose, void* stream) {
    if (!x || !codes || !descale || !aligned16(x) || !aligned16(codes) || !aligned4(descale))
        return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || N > kMaxLen || (long long)B * H > kMaxHeads)
        return ATTN_ERR_INVALID_ARG;
    if (transpose != 0 && transpose != 1) return ATTN_ERR_INVALID_ARG;
    if ((long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;  // grid.y
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    DeviceInfo dev;
    attn_status_t st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    return launch_fp8_quantize(x, codes, descale, signs, B * H, N, transpose,
                               static_cast<cudaStream_t>(stream), dev);
}

attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                           const float* k_descale, const float* v_descale, void* o, float* lse,
                           int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                           int rotated, attn_out_dtype_t o_dtype, void* stream) {
    if (!q_descale || !k_descale || !v_descale || !aligned4(q_descale) || !aligned4(k_descale) ||
        !aligned4(v_descale))
        return ATTN_ERR_INVALID_ARG;
    if (rotated != 0 && rotated != 1) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_fwd(q8, k8, vt8, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, o_dtype);
    if (st != ATTN_OK) return st;
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    // Q and K rotated by the same signed Hadamard matrix H (entries +-1, H H^T
    // = d I): (Q D H)(K D H)^T = d Q K^T, so the scores carry a factor d that
    // the scale takes back (exact: d = 128 is a power of two).
    const float eff = rotated ? scale / (float)d : scale;
    return launch_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk,
                          causal, eff, o_dtype, static_cast<cudaStream_t>(stream), dev);
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int total_q, int total_k, int max_seqlen_q,
                              int max_seqlen_k, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, void* stream) {
    if (!cu_seqlens_q || !cu_seqlens_k || !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k))
        return ATTN_ERR_INVALID_ARG;
    if (total_q < 1 || total_k < 1 || total_q > kMaxPackedRows || total_k > kMaxPackedRows)
        return ATTN_ERR_INVALID_ARG;
    if (max_seqlen_q > total_q || max_seqlen_k > total_k) return ATTN_ERR_INVALID_ARG;
    // (the per-sequence causal condition is checked on the device)
    attn_status_t st = check_fwd(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, d, 0,
                                 scale, o_dtype);
    if (st != ATTN_OK) return st;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!fwd_head_dim_supported(d)) return ATTN_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    if (d > 128)
        return launch_fwd_wide_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv,
                                      total_q, total_k, max_seqlen_q, max_seqlen_k, d, causal,
                                      scale, o_dtype, static_cast<cudaStream_t>(stream), dev);
    return launch_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                             total_k, max_seqlen_q, max_seqlen_k, d, causal, scale, o_dtype,
                             static_cast<cudaStream_t>(stream), dev);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
    if (check_common(B, Hq, Hkv, d, 1.0f, ATTN_OUT_BF16) != ATTN_OK) return 0;
    if (Nq < 1 || Nk < 1 || Nq > kMaxLen || Nk > kMaxLen) return 0;
    if (!fwd_head_dim_supported(d)) return 0;
    return bwd_workspace_bytes(B, Hq, Nq, d);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                       attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype, void* workspace,
                       size_t workspace_bytes, void* stream) {
    attn_status_t st = check_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, o_dtype);
    if (st != ATTN_OK) return st;
    // (check_fwd has limited d to the forward's head dims, which the backward takes too)
    if (!dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return ATTN_ERR_INVALID_ARG;
    if (grad_dtype != ATTN_OUT_BF16 && grad_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
    const size_t need = bwd_workspace_bytes(B, Hq, Nq, d);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    return launch_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, causal, scale,
                      o_dtype, grad_dtype, workspace, static_cast<cudaStream_t>(stream), dev);
}

size_t attn_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int d) {
    if (check_common(B, Hq, Hkv, d, 1.0f, ATTN_OUT_BF16) != ATTN_OK) return 0;
    if (total_q < 1 || total_q > kMaxPackedRows || !fwd_head_dim_supported(d)) return 0;
    return bwd_varlen_workspace_bytes(B, Hq, total_q);
}

attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int total_q, int total_k, int max_seqlen_q,
                              int max_seqlen_k, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (!cu_seqlens_q || !cu_seqlens_k || !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k))
        return ATTN_ERR_INVALID_ARG;
    if (total_q < 1 || total_k < 1 || total_q > kMaxPackedRows || total_k > kMaxPackedRows)
        return ATTN_ERR_INVALID_ARG;
    if (max_seqlen_q > total_q || max_seqlen_k > total_k) return ATTN_ERR_INVALID_ARG;
    // (the per-sequence causal condition is checked on the device)
    attn_status_t st = check_fwd(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, d, 0,
                                 scale, o_dtype);
    if (st != ATTN_OK) return st;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return ATTN_ERR_INVALID_ARG;
    if (grad_dtype != ATTN_OUT_BF16 && grad_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
    if (!fwd_head_dim_supported(d)) return ATTN_ERR_UNSUPPORTED;
    const size_t need = bwd_varlen_workspace_bytes(B, Hq, total_q);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    return launch_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, Hq,
                             Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, causal, scale,
                             o_dtype, grad_dtype, workspace, static_cast<cudaStream_t>(stream), dev);
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nmax, int d, int num_splits) {
    if (check_decode_shape(B, Hq, Hkv, Nmax, d, num_splits) != ATTN_OK) return 0;
    int sms = 0;
    if (current_num_sms(&sms) != 0) return 0;
    const int chunk = decode_chunk(Nmax, B, Hkv, sms, num_splits);
    return decode_workspace_bytes(B, Hq, Nmax, decode_pad_head_dim(d), chunk);
}

int attn_decode_kernel_launches(int B, int Hq, int Hkv, int Nmax, int d, int num_splits) {
    if (check_decode_shape(B, Hq, Hkv, Nmax, d, num_splits) != ATTN_OK) return -1;
    int sms = 0;
    if (current_num_sms(&sms) != 0) return -1;
    const int chunk = decode_chunk(Nmax, B, Hkv, sms, num_splits);
    const int max_splits = (Nmax + chunk - 1) / chunk;
    return decode_merges_in_kernel(B, Hkv, Hq / Hkv, max_splits, decode_pad_head_dim(d)) ? 1 : 2;
}

attn_status_t attn_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nmax, int d, float scale, int num_splits, void* workspace,
                          size_t workspace_bytes, attn_out_dtype_t o_dtype, void* stream) {
    attn_status_t st = check_decode_call(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Nmax,
                                         d, scale, num_splits, o_dtype);
    if (st != ATTN_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    const int chunk = decode_chunk(Nmax, B, Hkv, dev.num_sms, num_splits);
    const size_t need = decode_workspace_bytes(B, Hq, Nmax, decode_pad_head_dim(d), chunk);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    return launch_decode(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Nmax, d, scale, chunk,
                         workspace, o_dtype, static_cast<cudaStream_t>(stream), dev);
}

attn_status_t attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                const int* block_table, const int* seqlens, void* o, float* lse,
                                int B, int Hq, int Hkv, long long num_blocks, int page_size,
                                int max_blocks, int d, float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, attn_out_dtype_t o_dtype, void* stream) {
    if (!q || !k_pages || !v_pages || !block_table || !seqlens || !o) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
        !aligned4(seqlens) || !aligned4(block_table))
        return ATTN_ERR_INVALID_ARG;
    if (lse && !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
    if (num_blocks < 1 || max_blocks < 1 || page_size < 64) return ATTN_ERR_INVALID_ARG;
    if (page_size % 64 != 0) return ATTN_ERR_UNSUPPORTED;
    if ((long long)max_blocks * page_size > kMaxLen || num_blocks >= (1ll << 31))
        return ATTN_ERR_INVALID_ARG;
    const int Nmax = max_blocks * page_size;
    attn_status_t st = check_common(B, Hq, Hkv, d, scale, o_dtype);
    if (st != ATTN_OK) return st;
    if ((st = check_decode_shape(B, Hq, Hkv, Nmax, d, num_splits)) != ATTN_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != ATTN_OK) return st;
    const int chunk = decode_chunk(Nmax, B, Hkv, dev.num_sms, num_splits);
    const size_t need = decode_workspace_bytes(B, Hq, Nmax, decode_pad_head_dim(d), chunk);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
    return launch_decode_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, B, Hq, Hkv,
                               num_blocks, page_size, max_blocks, d, scale, chunk, workspace,
                               o_dtype, static_cast<cudaStream_t>(stream), dev);
}

const char* attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    }
    return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_selftest_bounded_wait(int mode, int* result, void* stream) {
    if ((mode != 0 && mode != 1) || !result || !aligned4(result)) return ATTN_ERR_INVALID_ARG;
    DeviceInfo dev;
    attn_status_t st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    attn_selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(mode, result, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_last_device_error(void* stream) {
    DeviceInfo dev;
    attn_status_t st = current_device_info(&dev);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, dev.err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const unsigned int zero = 0;
    if (word != 0 && cudaMemcpy(dev.err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word & kErrTimeout) return ATTN_ERR_TIMEOUT;
    if (word & kErrLayout) return ATTN_ERR_CUDA;
    if (word & kErrBadSeqlen) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int attn_decode_num_splits(int units, int num_sms, int max_splits) {
    if (units < 1 || num_sms < 1 || max_splits < 1) return 0;
    std::vector<double> eff((size_t)max_splits + 1, 0.0);
    double best = 0.0;
    for (int s = 1; s <= max_splits; ++s) {
        const double waves = (double)units * s / num_sms;
        eff[s] = waves / std::ceil(waves);
        best = std::max(best, eff[s]);
    }
    for (int s = 1; s <= max_splits; ++s)
        if (eff[s] >= 0.85 * best) return s;
    return 1;
}

long long attn_list_schedule(const int* costs, int n, int workers, int lpt, long long* loads_out) {
    if (n < 0 || workers < 1 || (n > 0 && !costs)) return -1;
    std::vector<int> order((size_t)n);
    std::iota(order.begin(), order.end(), 0);
    if (lpt)
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int b) { return costs[a] > costs[b]; });
    std::vector<long long> load((size_t)workers, 0);
    for (int idx : order) {
        if (costs[idx] < 0) return -1;
        int w = 0;
        for (int i = 1; i < workers; ++i)
            if (load[i] < load[w]) w = i;
        load[w] += costs[idx];
    }
    if (loads_out) std::copy(load.begin(), load.end(), loads_out);
    return workers ? *std::max_element(load.begin(), load.end()) : 0;
}

int attn_kv_tiles(int row0, int rows, int Nq, int Nk, int causal, int block) {
    return kv_tiles_for_rows(row0, rows, Nq, Nk, causal, block);
}

long long attn_fwd_num_units(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1 || Hq % Hkv) return -1;
    return make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal).units;
}

int attn_fwd_schedule(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms,
                      long long n, int* units_out, int* cost_out) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1 || Hq % Hkv || !units_out ||
        num_sms < 0)
        return -1;
    const FwdShape s = make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal, num_sms);
    if (n != s.units || s.units >= (1ll << 31)) return -1;
    for (long long i = 0; i < n; ++i) {
        int bh, mb;
        unit_of(s, (uint32_t)i, bh, mb);
        units_out[3 * i] = bh / Hq;
        units_out[3 * i + 1] = bh % Hq;
        units_out[3 * i + 2] = mb;
        if (cost_out) cost_out[i] = tile_kv_count(mb, 0, s) + tile_kv_count(mb, 1, s);
    }
    return 0;
}

int attn_fwd_split_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms,
                        int* n_full, int* n_split, int* parts) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1 || Hq % Hkv || num_sms < 1 ||
        !n_full || !n_split || !parts)
        return -1;
    const FwdShape s = make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal);
    if (s.units >= (1ll << 31)) return -1;
    const FwdSplit sp = plan_tail_split(s, num_sms);
    *n_full = sp.n_full;
    *n_split = sp.n_split;
    *parts = sp.parts;
    return 0;
}

}  // extern "C"
