// attn_fp8_sm103.cu -- FP8 (E4M3) forward for sm_103a: block quantization with
// an optional random-sign Hadamard rotation, and the fused attention forward
// on E4M3 operands.
//
// Method: lecture notes "Optimizing Attention for Modern Hardware:
// FlashAttention 1-4", 4.4 (FP8 tensor cores, block quantization, incoherent
// processing with a random-sign Hadamard matrix, V laid out for the 8-bit
// MMA); "Flash Attention 3/4 notes", FA3 section 2 (one scale per block,
// (QM)(KM)^T = QK^T).
//
// attn_fp8_quantize_rows_kernel / attn_fp8_quantize_kernel (HBM-bound): one
//   CTA per (batch * head, block of 128 rows).  With signs given, a row x
//   becomes H (s o x) (H the unnormalised Sylvester-Hadamard matrix) by the
//   fast Walsh-Hadamard transform in fp32: stages h = 1, 2, ..., 64; each pair
//   (i, i + h) becomes (a + b, a - b); the stages inside a lane's slice of the
//   row run in registers, the others through shuffles.  The block's amax gives
//   inv = 448 / amax and descale = amax / 448; codes are E4M3(x * inv), written
//   row-major [B, H, N, 128] by the rows kernel (16 entries per lane, values
//   kept in registers) or, for V, transposed [B, H, 128, Np] by the other
//   (the block staged in shared memory) so that the P.V product reads V
//   K-major.
//
// attn_fwd_fp8_kernel (tensor-bound): the bf16 forward's persistent design
//   (one CTA per SM, device-side queue over the units of fwd_sched.h, warp 0
//   TMA producer, warp 1 MMA issuer, two softmax warpgroups of one Q tile each)
//   with 8-bit tiles: S = Q K^T and O += P V on tcgen05 kind::f8f6f4 (K = 32
//   per instruction), P written to TMEM as E4M3 (4 keys per column).  The
//   block scales enter the softmax per KV tile: the score of key j is
//   s * c_j with c_j = scale * sq * sk_j * log2(e), and the probabilities are
//   kept in a frame that absorbs V's block scale sv_j:
//     P~ = 2^(s c_j + log2 sv_j - m + 4),   O_acc = sum P~ V8,
//     l = sum_j (sum P~) / sv_j,            O = O_acc / l,
//   with one running max m of s c_j + log2 sv_j, raised when a tile's max
//   passes it by more than tau = 4 (so P~ <= 2^8 fits E4M3), and the same two
//   row sums as the bf16 forward (the unrounded one for the LSE, the other
//   carrying the rounding of each tile's largest P~).
//   LSE = ln2 * (m - 4 + log2 lx).  d = 128 only.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "fwd_sched.h"

namespace gb300 {
namespace {

constexpr int kD = 128;
constexpr float kE4m3Max = 448.0f;
constexpr float kTau8 = 4.0f;        // rescale threshold (log2 units)
constexpr float kLift = 4.0f;        // P~ = 2^(x - m + kLift) <= 2^(tau + lift) = 256
constexpr float kLn2f = 0.69314718055994530942f;
constexpr float kLog2ef = 1.44269504088896340736f;

// ---------------------------------------------------------------------------
// Quantization
// ---------------------------------------------------------------------------
constexpr int kQThreads = 128;
constexpr int kQSmem = 128 * kD * 4;  // the block's 128 rows in fp32

// One butterfly stage between lanes: pairs (i, i + h) with h = 4 * bit; the
// lane holding i keeps a + b, the lane holding i + h keeps a - b.
__device__ __forceinline__ float fwht_xlane(float v, int lane, int bit) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, v, bit);
    return (lane & bit) ? __fsub_rn(o, v) : __fadd_rn(v, o);
}

template <bool ROTATE, bool TRANSPOSE>
__global__ void __launch_bounds__(kQThreads)
attn_fp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ out,
                         float* __restrict__ descale, const int8_t* __restrict__ signs, int N,
                         int npad, int nblk) {
    extern __shared__ __align__(16) float tile[];  // [128][kD]
    __shared__ float warp_max[4];
    const int blk = blockIdx.x;
    const long long bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float sg[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (ROTATE) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sg[e] = (float)__ldg(signs + 4 * lane + e);
    }
    float amax = 0.f;
    // all 32 rows' loads first (8 KiB in flight per warp), then the arithmetic
    uint2 raw[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int row = blk * 128 + warp * 32 + i;
        raw[i] = row < N ? __ldg(reinterpret_cast<const uint2*>(x + (bh * N + row) * kD) + lane)
                         : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int r = warp * 32 + i;
        float v[4];
        v[0] = __uint_as_float(raw[i].x << 16);
        v[1] = __uint_as_float(raw[i].x & 0xFFFF0000u);
        v[2] = __uint_as_float(raw[i].y << 16);
        v[3] = __uint_as_float(raw[i].y & 0xFFFF0000u);
        if constexpr (ROTATE) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(v[e], sg[e]);
            // h = 1: (0,1), (2,3); h = 2: (0,2), (1,3)
            float a0 = __fadd_rn(v[0], v[1]), a1 = __fsub_rn(v[0], v[1]);
            float a2 = __fadd_rn(v[2], v[3]), a3 = __fsub_rn(v[2], v[3]);
            v[0] = __fadd_rn(a0, a2); v[2] = __fsub_rn(a0, a2);
            v[1] = __fadd_rn(a1, a3); v[3] = __fsub_rn(a1, a3);
#pragma unroll
            for (int bit = 1; bit < 32; bit <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = fwht_xlane(v[e], lane, bit);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(v[e]));
        *reinterpret_cast<float4*>(tile + r * kD + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(warp_max[0], warp_max[1]), fmaxf(warp_max[2], warp_max[3]));
    const float inv = amax > 0.f ? __fdiv_rn(kE4m3Max, amax) : 0.f;
    if (threadIdx.x == 0) descale[bh * nblk + blk] = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
    if constexpr (!TRANSPOSE) {
        for (int i = 0; i < 32; ++i) {
            const int r = warp * 32 + i;
            const int row = blk * 128 + r;
            if (row >= N) break;
            const float4 t = *reinterpret_cast<const float4*>(tile + r * kD + 4 * lane);
            const uint32_t w = pack_e4m3x2(__fmul_rn(t.x, inv), __fmul_rn(t.y, inv)) |
                               (pack_e4m3x2(__fmul_rn(t.z, inv), __fmul_rn(t.w, inv)) << 16);
            reinterpret_cast<uint32_t*>(out + (bh * N + row) * kD)[lane] = w;
        }
    } else {
        // thread c writes row c of V^T: keys blk*128 + [0, 128) (16 per store)
        const int c = threadIdx.x;
        uint8_t* dst = out + (bh * kD + c) * (long long)npad + (long long)blk * 128;
        for (int k0 = 0; k0 < 128; k0 += 16) {
            if (blk * 128 + k0 >= npad) break;  // npad is a multiple of 16
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = k0 + 4 * q + e;
                    f[e] = blk * 128 + key < N ? __fmul_rn(tile[key * kD + c], inv) : 0.f;
                }
                w[q] = pack_e4m3x2(f[0], f[1]) | (pack_e4m3x2(f[2], f[3]) << 16);
            }
            *reinterpret_cast<uint4*>(dst + k0) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Row-major output (Q, K): 256 threads, a warp takes 16 rows, four at a time
// (8 lanes per row, 16 consecutive entries per lane), so the butterfly stages
// h = 1 .. 8 stay inside a lane and only h = 16, 32, 64 cross lanes; the values
// stay in registers between the amax and the codes.
constexpr int kRThreads = 256;

template <bool ROTATE>
__global__ void __launch_bounds__(kRThreads)
attn_fp8_quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ out,
                              float* __restrict__ descale, const int8_t* __restrict__ signs,
                              int N, int nblk) {
    __shared__ float warp_max[8];
    const int blk = blockIdx.x;
    const long long bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 3, pos = lane & 7;   // row within a group of 4, 16-entry slice
    uint4 raw[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = blk * 128 + warp * 16 + 4 * i + g;
        const uint4* src = reinterpret_cast<const uint4*>(x + (bh * N + row) * kD + 16 * pos);
        raw[i][0] = row < N ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
        raw[i][1] = row < N ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
    float sg[16];
    if constexpr (ROTATE) {
#pragma unroll
        for (int e = 0; e < 16; ++e) sg[e] = (float)__ldg(signs + 16 * pos + e);
    }
    float v[4][16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[8] = {raw[i][0].x, raw[i][0].y, raw[i][0].z, raw[i][0].w,
                               raw[i][1].x, raw[i][1].y, raw[i][1].z, raw[i][1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            v[i][2 * e] = __uint_as_float(w[e] << 16);
            v[i][2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
        if constexpr (ROTATE) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[i][e] = __fmul_rn(v[i][e], sg[e]);
#pragma unroll
            for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    if (e & h) continue;
                    const float a = v[i][e], b = v[i][e + h];
                    v[i][e] = __fadd_rn(a, b);
                    v[i][e + h] = __fsub_rn(a, b);
                }
            }
#pragma unroll
            for (int bit = 1; bit < 8; bit <<= 1) {   // h = 16 * bit
#pragma unroll
                for (int e = 0; e < 16; ++e) v[i][e] = fwht_xlane(v[i][e], lane, bit);
            }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[i][e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) amax = fmaxf(amax, warp_max[k]);
    const float inv = amax > 0.f ? __fdiv_rn(kE4m3Max, amax) : 0.f;
    if (threadIdx.x == 0) descale[bh * nblk + blk] = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = blk * 128 + warp * 16 + 4 * i + g;
        if (row >= N) continue;
        uint32_t c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            c[q] = pack_e4m3x2(__fmul_rn(v[i][4 * q], inv), __fmul_rn(v[i][4 * q + 1], inv)) |
                   (pack_e4m3x2(__fmul_rn(v[i][4 * q + 2], inv), __fmul_rn(v[i][4 * q + 3], inv)) << 16);
        *reinterpret_cast<uint4*>(out + (bh * N + row) * kD + 16 * pos) = make_uint4(c[0], c[1], c[2], c[3]);
    }
}

// ---------------------------------------------------------------------------
// Attention on E4M3 operands
// ---------------------------------------------------------------------------
constexpr int kThreads = 384;
constexpr int kRegsControl = 104;
constexpr int kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr uint32_t kNegInf = 0xFF800000u;

struct Cfg8 {
    static constexpr int kTileBytes = 128 * 128;           // 128 rows x 128 bytes
    static constexpr int kStages = 8;                      // K / V^T ring slots
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kStgOff = kRingOff + kStages * kTileBytes;
    static constexpr int kStgBytesPerWarp = 2 * 2048;
    static constexpr int kBarOff = kStgOff + 8 * kStgBytesPerWarp;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static __host__ __device__ constexpr uint32_t col_s(int t) { return uint32_t(t) * 128u; }
    static __host__ __device__ constexpr uint32_t col_o(int t) { return 256u + uint32_t(t) * kD; }
};

struct Fp8Params {
    FwdShape shape;
    int group;
    int off;            // Nk - Nq
    float scale;        // softmax scale (already divided by d for rotated Q, K)
    uint32_t slot;
    int nblk_q, nblk_k; // 128-row blocks per head of Q / of K and V
    const float* q_descale;
    const float* k_descale;
    const float* v_descale;
};

constexpr uint32_t kQueueSlots8 = 256;
__device__ unsigned int g_fp8_queue[kQueueSlots8][2];  // ticket counter, exit count

struct Item8 {
    int bh, mb, e[2];
};

struct __align__(8) Bars8 {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2];
    uint64_t unit_full[2], unit_empty[2];
    uint64_t drain;
    Item8 item[2];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars8) <= Cfg8::kBarBytes, "barrier block");

constexpr int kConsumers8 = 9;

__device__ __forceinline__ bool take_item8(Bars8* bars, uint32_t k, Item8& w,
                                           const volatile int* abort_flag) {
    const uint32_t i = k & 1u;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_full[i]), (k >> 1) & 1u, abort_flag)))
        return false;
    const volatile Item8* src = &bars->item[i];
    w.bh = src->bh;
    w.mb = src->mb;
    w.e[0] = src->e[0];
    w.e[1] = src->e[1];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars->unit_empty[i]));
    return true;
}

__device__ __forceinline__ void raise_abort8(Bars8* bars, unsigned int* err) {
    atomicOr(err, kErrTimeout);
    *((volatile int*)&bars->abort) = 1;
}

__device__ void run_producer8(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              uint8_t* smem, Bars8* bars, const Fp8Params& p, unsigned int* err) {
    using C = Cfg8;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1;
    unsigned int* queue = g_fp8_queue[p.slot];
    uint32_t q_issued[2] = {0u, 0u};
    long long L = 0;
    bool ok = true;
    for (int local = 0; ok; ++local) {
        const uint32_t hs = (uint32_t)local & 1u;
        if (local >= 2)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_empty[hs]),
                                                   (uint32_t)((local >> 1) - 1) & 1u, abort_flag));
        if (!ok) break;
        uint32_t u = blockIdx.x;
        if (local > 0) {
            if (leader) u = gridDim.x + atomicAdd(&queue[0], 1u);
            u = __shfl_sync(0xFFFFFFFFu, u, leader_lane);
        }
        const bool done = u >= (uint32_t)s.units;
        int bh = -1, mb = 0, n0 = 0, n1 = 0;
        if (!done) {
            unit_of(s, u, bh, mb);
            n0 = tile_kv_count(mb, 0, s);
            n1 = tile_kv_count(mb, 1, s);
        }
        if (leader) {
            volatile Item8* dst = &bars->item[hs];
            dst->bh = bh;
            dst->mb = mb;
            dst->e[0] = n0;
            dst->e[1] = n1;
            mbar_arrive(smem_u32(&bars->unit_full[hs]));
        }
        __syncwarp();
        if (done) break;
        const int b = bh / s.Hq;
        const int hq = bh - b * s.Hq;
        const int bkv = b * s.Hkv + hq / p.group;
        const int j1 = n0 > n1 ? n0 : n1;
        for (int t = 0; t < 2 && ok; ++t) {
            if (local > 0)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->q_empty[t]), (local - 1) & 1, abort_flag));
            if (!ok) break;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->q_full[t]);
                mbar_arrive_expect_tx(bar, C::kTileBytes);
                tma_load_3d(smem_u32(smem + t * C::kTileBytes), tq, bar, 0, mb * kUnitRows + t * kTileM, bh);
            }
            __syncwarp();
            ++q_issued[t];
        }
        for (int j = 0; j < j1 && ok; ++j) {
#pragma unroll 1
            for (int which = 0; which < 2; ++which) {
                const int slot = (int)(L % C::kStages);
                const long long round = L / C::kStages;
                if (round > 0)
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->kv_empty[slot]),
                                                           (uint32_t)((round - 1) & 1), abort_flag));
                if (!ok) break;
                if (leader) {
                    const uint32_t bar = smem_u32(&bars->kv_full[slot]);
                    mbar_arrive_expect_tx(bar, C::kTileBytes);
                    const uint32_t dst = smem_u32(smem + C::kRingOff + slot * C::kTileBytes);
                    if (which == 0)
                        tma_load_3d(dst, tk, bar, 0, kTileN * j, bkv);        // K: keys x d
                    else
                        tma_load_3d(dst, tv, bar, kTileN * j, 0, bkv);        // V^T: d x keys
                }
                __syncwarp();
                ++L;
            }
        }
    }
    if (!ok && leader) raise_abort8(bars, err);
    if (leader) {
        __threadfence();
        if (atomicAdd(&queue[1], 1u) == gridDim.x - 1) {
            queue[0] = 0u;
            queue[1] = 0u;
        }
    }
    for (int t = 0; t < 2; ++t)
        if (q_issued[t] > 0) mbar_wait(smem_u32(&bars->q_full[t]), (q_issued[t] - 1) & 1, nullptr);
    for (int slot = 0; slot < C::kStages && slot < L; ++slot) {
        const long long n_s = (L - slot + C::kStages - 1) / C::kStages;
        mbar_wait(smem_u32(&bars->kv_full[slot]), (uint32_t)((n_s - 1) & 1), nullptr);
    }
    __syncwarp();
}

constexpr uint32_t kDescHi8 = sdesc_hi_sw128(1024);

// S_t = Q_t K^T: 4 steps of 32 bytes along a 128-byte swizzled row.
__device__ __forceinline__ void issue_qk8(uint32_t tmem, int t, uint32_t q_lo, uint32_t k_lo,
                                          uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ss_f8_warp(tmem + Cfg8::col_s(t), sdesc_join(q_lo + kk * (32 >> 4), kDescHi8),
                       sdesc_join(k_lo + kk * (32 >> 4), kDescHi8), idesc, kk > 0 ? 1u : 0u);
}

// O_t += P_t V: A = P (E4M3, 4 keys per TMEM column: 8 columns per 32 keys),
// B = V^T tile (d rows x 128 keys, K-major).
__device__ __forceinline__ void issue_pv8(uint32_t tmem, int t, uint32_t v_lo, uint32_t idesc,
                                          bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ts_f8_warp(tmem + Cfg8::col_o(t), tmem + Cfg8::col_s(t) + kk * 8,
                       sdesc_join(v_lo + kk * (32 >> 4), kDescHi8), idesc,
                       (accumulate || kk > 0) ? 1u : 0u);
}

__device__ void run_mma8(uint8_t* smem, Bars8* bars, uint32_t tmem, unsigned int* err) {
    using C = Cfg8;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idesc = make_idesc_e4m3(128, 128);
    const uint32_t q_lo[2] = {sdesc_lo(smem_u32(smem), 16), sdesc_lo(smem_u32(smem + C::kTileBytes), 16)};
    const uint32_t ring = smem_u32(smem + C::kRingOff);
    auto lo = [&](int slot) { return sdesc_lo(ring + slot * C::kTileBytes, 16); };
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag));
    };
    long long Cn = 0;
    uint32_t cnt_p[2] = {0u, 0u};
    bool ok = true;
    for (int local = 0; ok; ++local) {
        Item8 w;
        ok = take_item8(bars, (uint32_t)local, w, abort_flag);
        if (!ok || w.bh < 0) break;
        const int n[2] = {w.e[0], w.e[1]};
        const int j1 = n[0] > n[1] ? n[0] : n[1];
        for (int t = 0; t < 2 && ok; ++t) ok = wait_all(smem_u32(&bars->q_full[t]), local & 1);
        if (!ok) break;
        int slot_k = (int)(Cn % C::kStages);
        ok = wait_all(smem_u32(&bars->kv_full[slot_k]), (uint32_t)((Cn / C::kStages) & 1));
        ++Cn;
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
            if (n[t] > 0) {
                issue_qk8(tmem, t, q_lo[t], lo(slot_k), idesc);
                mma_commit_warp(smem_u32(&bars->s_full[t]));
            }
            if (n[t] <= 1) mma_commit_warp(smem_u32(&bars->q_empty[t]));
        }
        mma_commit_warp(smem_u32(&bars->kv_empty[slot_k]));
        for (int j = 0; j < j1 && ok; ++j) {
            const int slot_v = (int)(Cn % C::kStages);
            ok = wait_all(smem_u32(&bars->kv_full[slot_v]), (uint32_t)((Cn / C::kStages) & 1));
            ++Cn;
            if (!ok) break;
            tc_fence_after();
            bool k_ready = false;
            for (int t = 0; t < 2 && ok; ++t) {
                if (j >= n[t]) continue;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->p_full[t]), cnt_p[t] & 1, abort_flag, 32));
                ++cnt_p[t];
                if (!ok) break;
                tc_fence_after();
                issue_pv8(tmem, t, lo(slot_v), idesc, j > 0);
                if (j + 1 < n[t]) {
                    if (!k_ready) {
                        slot_k = (int)(Cn % C::kStages);
                        ok = wait_all(smem_u32(&bars->kv_full[slot_k]), (uint32_t)((Cn / C::kStages) & 1));
                        ++Cn;
                        if (!ok) break;
                        tc_fence_after();
                        k_ready = true;
                    }
                    issue_qk8(tmem, t, q_lo[t], lo(slot_k), idesc);
                    mma_commit_warp(smem_u32(&bars->s_full[t]));
                    if (j + 2 == n[t]) mma_commit_warp(smem_u32(&bars->q_empty[t]));
                } else {
                    mma_commit_warp(smem_u32(&bars->o_full[t]));
                }
            }
            if (!ok) break;
            mma_commit_warp(smem_u32(&bars->kv_empty[slot_v]));
            if (k_ready) mma_commit_warp(smem_u32(&bars->kv_empty[slot_k]));
        }
    }
    if (!ok && leader) raise_abort8(bars, err);
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// One KV tile of the softmax for this thread's row (see the file header):
// c = scale * sq * sk_j * log2 e, lv = log2 sv_j, isv = 1 / sv_j.
template <bool MASKED>
__device__ __forceinline__ void softmax_tile8(uint32_t (&sr)[128], int lim, bool first, float c,
                                              float lv, float isv, uint32_t tS, uint32_t tO,
                                              float& m, float& l, float& lx) {
    if constexpr (MASKED) {
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
            if (cc > lim) sr[cc] = kNegInf;
    }
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 128; cc += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[cc + 4]), __uint_as_float(sr[cc + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[cc + 6]), __uint_as_float(sr[cc + 7]));
    }
    const float smax = fmax3(fmaxf(mx0, mx1), mx2, mx3);
    const float mt = fmaf(smax, c, lv);
    const bool need = mt > m + kTau8;
    if (__any_sync(0xFFFFFFFFu, need)) {
        const float m_new = fmaxf(m, mt);
        const float alpha = ex2(m - m_new);
        l *= alpha;
        lx *= alpha;
        if (!first) {
            const uint64_t a2 = f2(alpha, alpha);
#pragma unroll 1
            for (int cc = 0; cc < kD; cc += 32) {
                uint32_t r[32];
                tmem_ld32(tO + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float a, b;
                    f2_split(f2_mul(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), a2), a, b);
                    r[i] = __float_as_uint(a);
                    r[i + 1] = __float_as_uint(b);
                }
                tmem_st32(tO + cc, r);
            }
        }
        m = m_new;
    }
    // P~ = 2^(s c + lv - m + lift); the largest one's E4M3 rounding error
    const float bias = lv - m + kLift;
    const float pmax = ex2(fmaf(smax, c, bias));
    const float corr = e4m3_round_f32(pmax) - pmax;
    const uint64_t c2 = f2(c, c), b2 = f2(bias, bias);
    uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int col = half * 64 + 4 * i;
            float x0, x1, x2, x3;
            f2_split(f2_fma(f2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), c2, b2), x0, x1);
            f2_split(f2_fma(f2(__uint_as_float(sr[col + 2]), __uint_as_float(sr[col + 3])), c2, b2), x2, x3);
            float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            if constexpr (MASKED) {
                p0 = col <= lim ? p0 : 0.f;
                p1 = col + 1 <= lim ? p1 : 0.f;
                p2 = col + 2 <= lim ? p2 : 0.f;
                p3 = col + 3 <= lim ? p3 : 0.f;
            }
            pk[i] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
            if (i & 1) {
                acc0 = f2_add(acc0, f2(p0, p1));
                acc1 = f2_add(acc1, f2(p2, p3));
            } else {
                acc2 = f2_add(acc2, f2(p0, p1));
                acc3 = f2_add(acc3, f2(p2, p3));
            }
        }
        tmem_st16(tS + half * 16, pk);
    }
    float a, b;
    f2_split(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a, b);
    const float tsum = a + b;
    lx = fmaf(tsum, isv, lx);
    l = fmaf(tsum + corr, isv, l);
}

template <bool OUT_F32>
__device__ __forceinline__ void store_o_cols8(const float (&v)[32], int cc, uint8_t* stg,
                                              uint32_t& epi_buf, int lane, const CUtensorMap* to,
                                              int row0, int bh) {
    constexpr int kCols = OUT_F32 ? 16 : 32;
#pragma unroll
    for (int h = 0; h < 32 / kCols; ++h) {
        uint8_t* buf = stg + (epi_buf & 1) * 2048;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t dst = smem_u32(buf) + lane * 64;
        if constexpr (OUT_F32) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sts128(dst + 16 * i, __float_as_uint(v[h * 16 + 4 * i]), __float_as_uint(v[h * 16 + 4 * i + 1]),
                       __float_as_uint(v[h * 16 + 4 * i + 2]), __float_as_uint(v[h * 16 + 4 * i + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sts128(dst + 16 * i, pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                       pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(to, smem_u32(buf), cc + h * kCols, row0, bh);
            bulk_commit_group();
        }
        ++epi_buf;
    }
}

template <bool OUT_F32>
__device__ void run_softmax8(int t, int wq, int lane, uint8_t* smem, Bars8* bars, uint32_t tmem,
                             const Fp8Params& p, const CUtensorMap* to, float* __restrict__ lse_ptr,
                             unsigned int* err) {
    using C = Cfg8;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + C::col_s(t) + lane_off;
    const uint32_t tO = tmem + C::col_o(t) + lane_off;
    const uint32_t bar_s = smem_u32(&bars->s_full[t]);
    const uint32_t bar_p = smem_u32(&bars->p_full[t]);
    const uint32_t bar_o = smem_u32(&bars->o_full[t]);
    uint8_t* stg = smem + C::kStgOff + (t * 4 + wq) * C::kStgBytesPerWarp;
    uint32_t epi_buf = 0;
    uint32_t cnt_s = 0, cnt_o = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
        Item8 w;
        ok = take_item8(bars, k, w, abort_flag);
        if (!ok || w.bh < 0) break;
        const int bh = w.bh, mb = w.mb;
        const int n_t = t == 0 ? w.e[0] : w.e[1];
        if (n_t <= 0) continue;
        const int b = bh / s.Hq;
        const int hq = bh - b * s.Hq;
        const long long kvh = (long long)b * s.Hkv + hq / p.group;
        const float* skp = p.k_descale + kvh * p.nblk_k;
        const float* svp = p.v_descale + kvh * p.nblk_k;
        const float cq = p.scale * __ldg(p.q_descale + (long long)bh * p.nblk_q + mb * 2 + t) * kLog2ef;
        const int row = mb * kUnitRows + t * kTileM + wq * 32 + lane;
        int last_key = s.Nk - 1;
        if (s.causal) {
            const int lk = row + p.off;
            last_key = lk < last_key ? lk : last_key;
        }
        float m = -INFINITY, l = 0.f, lx = 0.f;
        float sk_n = __ldg(skp), sv_n = __ldg(svp);
        for (int j = 0; j < n_t; ++j) {
            const float sk = sk_n, sv = sv_n;
            if (j + 1 < n_t) {  // next tile's scales, in flight during this tile
                sk_n = __ldg(skp + j + 1);
                sv_n = __ldg(svp + j + 1);
            }
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s, cnt_s & 1, abort_flag, 32));
            ++cnt_s;
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
            tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
            tmem_wait_ld();
            const float c = cq * sk;
            const float lv = log2f(sv);
            const float isv = 1.0f / sv;
            const int lim = last_key - j * kTileN;
            if (__any_sync(0xFFFFFFFFu, lim < kTileN - 1))
                softmax_tile8<true>(sr, lim, j == 0, c, lv, isv, tS, tO, m, l, lx);
            else
                softmax_tile8<false>(sr, lim, j == 0, c, lv, isv, tS, tO, m, l, lx);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p);
        }
        if (!ok) break;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o, cnt_o & 1, abort_flag));
        ++cnt_o;
        if (!ok) break;
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const uint64_t il2 = f2(inv_l, inv_l);
        const int row0 = mb * kUnitRows + t * kTileM + wq * 32;
#pragma unroll 1
        for (int cc = 0; cc < kD; cc += 32) {
            uint32_t r[32];
            tmem_ld32(tO + cc, r);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2)
                f2_split(f2_mul(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), il2), v[i], v[i + 1]);
            store_o_cols8<OUT_F32>(v, cc, stg, epi_buf, lane, to, row0, bh);
        }
        if (row < s.Nq && lse_ptr)
            lse_ptr[(size_t)bh * s.Nq + (size_t)row] = (m - kLift + log2f(lx)) * kLn2f;
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
    if (!ok) raise_abort8(bars, err);
}

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    float* __restrict__ lse_ptr, const Fp8Params p, unsigned int* err) {
    using C = Cfg8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Bars8* bars = reinterpret_cast<Bars8*>(smem + C::kBarOff);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars->q_full[t]), 1);
            mbar_init(smem_u32(&bars->q_empty[t]), 1);
            mbar_init(smem_u32(&bars->s_full[t]), 1);
            mbar_init(smem_u32(&bars->p_full[t]), 4);
            mbar_init(smem_u32(&bars->o_full[t]), 1);
        }
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(smem_u32(&bars->kv_full[i]), 1);
            mbar_init(smem_u32(&bars->kv_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->unit_full[i]), 1);
            mbar_init(smem_u32(&bars->unit_empty[i]), kConsumers8);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&to);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (warp < 4) {
        reg_dealloc<kRegsControl>();
        if (warp == 0) run_producer8(&tq, &tk, &tv, smem, bars, p, err);
        if (warp == 1) run_mma8(smem, bars, tmem, err);
    } else {
        reg_alloc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        run_softmax8<OUT_F32>(t, warp & 3, lane, smem, bars, tmem, p, &to, lse_ptr, err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool OUT_F32>
attn_status_t launch_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, float* lse, const Fp8Params& p, int grid,
                           cudaStream_t stream, const DeviceInfo& dev) {
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_fwd_fp8_kernel<OUT_F32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg8::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    attn_fwd_fp8_kernel<OUT_F32><<<(unsigned)grid, kThreads, Cfg8::kSmemBytes, stream>>>(
        tq, tk, tv, to, lse, p, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <bool ROTATE, bool TRANSPOSE>
attn_status_t launch_quant_t(const void* x, void* out, float* descale, const int8_t* signs,
                             int BH, int N, int npad, int nblk, cudaStream_t stream,
                             const DeviceInfo& dev) {
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_fp8_quantize_kernel<ROTATE, TRANSPOSE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    dim3 grid((unsigned)nblk, (unsigned)BH);
    attn_fp8_quantize_kernel<ROTATE, TRANSPOSE><<<grid, kQThreads, kQSmem, stream>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(out), descale, signs, N, npad,
        nblk);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

attn_status_t launch_fp8_quantize(const void* x, void* out, float* descale, const int8_t* signs,
                                  int BH, int N, int transpose, cudaStream_t stream,
                                  const DeviceInfo& dev) {
    const int nblk = (N + 127) / 128;
    const int npad = (N + 15) / 16 * 16;
    if (!transpose) {
        dim3 grid((unsigned)nblk, (unsigned)BH);
        const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
        uint8_t* ob = static_cast<uint8_t*>(out);
        if (signs)
            attn_fp8_quantize_rows_kernel<true><<<grid, kRThreads, 0, stream>>>(xb, ob, descale, signs, N, nblk);
        else
            attn_fp8_quantize_rows_kernel<false><<<grid, kRThreads, 0, stream>>>(xb, ob, descale, signs, N, nblk);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    return signs ? launch_quant_t<true, true>(x, out, descale, signs, BH, N, npad, nblk, stream, dev)
                 : launch_quant_t<false, true>(x, out, descale, signs, BH, N, npad, nblk, stream, dev);
}

attn_status_t launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                             const float* k_descale, const float* v_descale, void* o, float* lse,
                             int B, int Hq, int Hkv, int Nq, int Nk, int causal, float scale,
                             attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev) {
    Fp8Params p;
    p.shape = make_fwd_shape(B, Hq, Hkv, Nq, Nk, kD, causal, dev.num_sms);
    if (p.shape.units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    p.group = Hq / Hkv;
    p.off = Nk - Nq;
    p.scale = scale;
    static std::atomic<uint32_t> launches{0};
    p.slot = launches.fetch_add(1u, std::memory_order_relaxed) % kQueueSlots8;
    p.nblk_q = (Nq + 127) / 128;
    p.nblk_k = (Nk + 127) / 128;
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    const long long units = p.shape.units;
    const int grid = (int)(units < dev.num_sms ? units : dev.num_sms);
    const int npad = (Nk + 15) / 16 * 16;
    CUtensorMap tq, tk, tv, to;
    attn_status_t st;
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if ((st = encode_tmap_u8_3d(&tq, q8, kD, kD, Nq, (long long)B * Hq, kD, kTileM)) != ATTN_OK) return st;
    if ((st = encode_tmap_u8_3d(&tk, k8, kD, kD, Nk, (long long)B * Hkv, kD, kTileN)) != ATTN_OK) return st;
    if ((st = encode_tmap_u8_3d(&tv, vt8, Nk, npad, kD, (long long)B * Hkv, kTileN, kD)) != ATTN_OK)
        return st;
    if ((st = encode_tmap_out_3d(&to, o, f32, kD, Nq, (long long)B * Hq, f32 ? 16 : 32, 32)) != ATTN_OK)
        return st;
    return f32 ? launch_fp8_t<true>(tq, tk, tv, to, lse, p, grid, stream, dev)
               : launch_fp8_t<false>(tq, tk, tv, to, lse, p, grid, stream, dev);
}

}  // namespace gb300
