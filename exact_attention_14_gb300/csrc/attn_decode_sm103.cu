// attn_decode_sm103.cu -- split-KV decode (Flash-Decoding) for sm_103a.
//
// Kernel 1 (split): one CTA per (split s, KV head g, sequence b).  It covers
// keys [s*chunk, min((s+1)*chunk, L_b)) of the valid prefix.  A producer warp
// streams 64-key K and V tiles with TMA into a 3-slot ring (128-byte swizzle);
// four consumer warps each take 16 keys of every tile.  The G = Hq/Hkv query
// heads that share KV head g are packed as the rows of a 16-row MMA tile
// (lecture notes "Optimizing Attention for Modern Hardware", 6.2 GQA
// packing), so every K/V byte is read from memory once for all G heads.
// Scores and P.V run on mma.sync (m16n8k16, bf16 in, fp32 accumulate); the
// online softmax (m, l) runs per row in fp32 registers; as in the forward, the
// sum of the bf16-rounded P normalises O and the sum of the unrounded P gives
// the LSE.  The four warps'
// partial results are merged in shared memory, and the CTA writes either the
// final O / LSE (when the sequence has one split) or a partial (o_s, lse_s)
// to the workspace.
//
// Merge of the splits: per (b, query head) with more than one split, the
// partials are merged by log-sum-exp: M = max lse_s, w_s = 2^(lse_s - M),
// O = sum w_s o_s / sum w_s, LSE = M + log2 sum w_s (lecture notes 6.1 and
// exercise 3; "FlashAttention tiling & online softmax" 7.1), in split order.
// Normally the last split CTA of a (b, KV head) to finish does it: each split
// CTA counts itself in on a per-(b, KV head) counter after writing its
// partial, and the one that completes the count merges the group's G heads
// and returns the counter to zero.  Shapes with more (b, KV head) groups than
// the counter table holds, or more splits than the merge's shared-memory
// scratch holds, use a second kernel (combine) for the merge.
//
// The decode path is memory-bound by design (it must read the KV cache once):
// it is measured against HBM bandwidth.  Keys at or past L_b are never used:
// their scores are masked by selection and their V rows are zeroed in shared
// memory before the P.V product, so NaN there cannot leak.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageKeys = 64;
constexpr int kDecStages = 3;
constexpr int kMaxGroup = 16;
constexpr int kAutoMaxChunk = 1024;  // keys; auto mode cuts sequences no coarser
constexpr float kLn2f = 0.69314718055994530942f;
constexpr float kLog2ef = 1.44269504088896340736f;

template <int D>
struct DecCfg {
    static constexpr int kHalfBytes = kStageKeys * D * 2;  // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kHalfBytes;
    static constexpr int kBarOff = kDecStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOff + 64 + 1024;
    // cross-warp merge scratch (reuses the stage ring once it is drained)
    static constexpr int kScratchO = 0;                                     // [4][16][D] f32
    static constexpr int kScratchM = kConsumerWarps * kMaxGroup * D * 4;    // [4][16] f32
    static constexpr int kScratchL = kScratchM + kConsumerWarps * kMaxGroup * 4;
    static constexpr int kScratchX = kScratchL + kConsumerWarps * kMaxGroup * 4;
    static_assert(kScratchX + kConsumerWarps * kMaxGroup * 4 <= kBarOff, "scratch fits");
};

struct DecParams {
    int B, Hq, Hkv, G, Nmax, chunk, max_splits;
    float c;   // scale * log2(e)
    int slot;  // arrival-counter slot of this launch; -1: merge in the combine kernel
    // paged cache (block_table != nullptr): the 64-key stage starting at key t of
    // sequence b lives in page block_table[b * max_blocks + t / page_size]
    const int* block_table;
    int page_size, max_blocks;
    int dh;    // the tensors' head dim (<= D: columns past dh are zeros in the tiles)
};

// Arrival counters of the in-kernel merge: one per (b, KV head) group and
// launch slot.  Launches rotate through the slots, and every count returns to
// zero when its group is merged, so up to kDecSlots launches may be in flight
// at the same time.
constexpr int kDecSlots = 64;
constexpr int kDecMaxGroups = 4096;
__device__ unsigned int g_dec_count[kDecSlots][kDecMaxGroups];

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk `ch` (0..D/8-1) of key row `key` inside a
// [64 keys x D] tile stored as D/64 boxes of 64x64 with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_off(int key, int ch) {
    return (uint32_t)((ch >> 3) * (kStageKeys * 128) + key * 128 + (((ch & 7) ^ (key & 7)) << 4));
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kDecThreads)
attn_decode_split_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         const __nv_bfloat16* __restrict__ q, const int* __restrict__ seqlens,
                         void* __restrict__ o, float* __restrict__ lse, float* __restrict__ ws_o,
                         float* __restrict__ ws_lse, const DecParams p, unsigned int* err) {
    using C = DecCfg<D>;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    int L = seqlens[b];
    if (L < 1 || L > p.Nmax) {
        if (split == 0 && g == 0 && threadIdx.x == 0) atomicOr(err, kErrBadSeqlen);
        L = L < 0 ? 0 : (L > p.Nmax ? p.Nmax : L);
    }
    const int t0 = split * p.chunk;
    if (t0 >= L) {  // uniform across the CTA: nothing started yet
        if (L == 0 && split == 0 && p.slot >= 0) {
            // an empty sequence: O = 0 and LSE = -inf for the group's heads
            for (int e = threadIdx.x; e < p.G * p.dh; e += blockDim.x) {
                const size_t bh = (size_t)b * p.Hq + (size_t)g * p.G + e / p.dh;
                const int col = e % p.dh;
                if constexpr (OUT_F32) static_cast<float*>(o)[bh * p.dh + col] = 0.f;
                else static_cast<__nv_bfloat16*>(o)[bh * p.dh + col] = __float2bfloat16_rn(0.f);
                if (col == 0 && lse) lse[bh] = -INFINITY;
            }
        }
        return;
    }
    const int t1 = min(t0 + p.chunk, L);
    const int n_stages = (t1 - t0 + kStageKeys - 1) / kStageKeys;
    const int nsplit_b = (L + p.chunk - 1) / p.chunk;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* empty = full + kDecStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kDecStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int kv_head = b * p.Hkv + g;
    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int st = 0; st < n_stages; ++st) {
                const int slot = st % kDecStages;
                if (st >= kDecStages) {
                    ok = mbar_wait(smem_u32(&empty[slot]), ((st / kDecStages) - 1) & 1, abort_flag);
                    if (!ok) break;
                }
                const uint32_t bar = smem_u32(&full[slot]);
                mbar_arrive_expect_tx(bar, C::kStageBytes);
                const uint32_t dk = smem_u32(smem + slot * C::kStageBytes);
                const uint32_t dv = dk + C::kHalfBytes;
                const int key = t0 + st * kStageKeys;
                if (p.block_table) {
                    // a page index out of range only reads zeros (TMA bounds checks)
                    const int blk = key / p.page_size;
                    const int page = __ldg(p.block_table + (size_t)b * p.max_blocks + blk);
                    const int off = key - blk * p.page_size;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_4d(dk + c * (kStageKeys * 128), &tk, bar, 64 * c, g, off, page);
                        tma_load_4d(dv + c * (kStageKeys * 128), &tv, bar, 64 * c, g, off, page);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        tma_load_3d(dk + c * (kStageKeys * 128), &tk, bar, 64 * c, key, kv_head);
                        tma_load_3d(dv + c * (kStageKeys * 128), &tv, bar, 64 * c, key, kv_head);
                    }
                }
                ++issued;
            }
            if (!ok) {
                atomicOr(err, kErrTimeout);
                *abort_flag = 1;
            }
            // drain: every issued copy lands before the CTA reuses or leaves smem
            for (int slot = 0; slot < kDecStages && slot < issued; ++slot) {
                const int n_s = (issued - slot + kDecStages - 1) / kDecStages;
                mbar_wait(smem_u32(&full[slot]), (n_s - 1) & 1, nullptr);
            }
        }
        __syncthreads();  // matches the consumers' barrier before the merge
        __syncthreads();
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int G = p.G;
    const int qr = lane >> 2, qc = lane & 3;
    // Query fragments (A operand, rows = packed heads of this KV group)
    uint32_t qa[D / 16][4];
    {
        // rows of the group's query heads; columns past dh are zero
        const int dh = p.dh;
        const __nv_bfloat16* qb = q + ((size_t)b * p.Hq + (size_t)g * G) * dh;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int c0 = ks * 16 + 2 * qc;
            const bool lo = c0 < dh, hi = c0 + 8 < dh;
            qa[ks][0] = (qr < G && lo) ? *reinterpret_cast<const uint32_t*>(qb + qr * dh + c0) : 0u;
            qa[ks][1] = (qr + 8 < G && lo) ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * dh + c0) : 0u;
            qa[ks][2] = (qr < G && hi) ? *reinterpret_cast<const uint32_t*>(qb + qr * dh + c0 + 8) : 0u;
            qa[ks][3] = (qr + 8 < G && hi) ? *reinterpret_cast<const uint32_t*>(qb + (qr + 8) * dh + c0 + 8) : 0u;
        }
    }
    float oacc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // rows qr, qr + 8 (log2 units)
    float l0 = 0.f, l1 = 0.f;              // per-thread sums of bf16-rounded P (normalise O)
    float x0 = 0.f, x1 = 0.f;              // per-thread sums of unrounded P (give the LSE)
    const float c = p.c;
    const int wk0 = warp * 16;
    bool ok = true;

    for (int st = 0; st < n_stages; ++st) {
        const int slot = st % kDecStages;
        // warp-uniform: ldmatrix and mma.sync below need every lane
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&full[slot]), (st / kDecStages) & 1, abort_flag));
        if (!ok) break;
        const int nvalid = min(kStageKeys, t1 - (t0 + st * kStageKeys));
        const uint32_t sK = smem_u32(smem + slot * C::kStageBytes);
        const uint32_t sV = sK + C::kHalfBytes;
        bool zeroed = false;
        if (wk0 < nvalid) {
            if (nvalid < wk0 + 16) {
                // zero this warp's V rows past the valid prefix (they may hold NaN)
                uint8_t* vrow0 = smem + slot * C::kStageBytes + C::kHalfBytes;
                const int first = nvalid;  // >= wk0
                const int rows = wk0 + 16 - first;
                for (int idx = lane; idx < rows * (D / 8); idx += 32) {
                    const int key = first + idx / (D / 8);
                    const int ch = idx % (D / 8);
                    *reinterpret_cast<uint4*>(vrow0 + swz_off(key, ch)) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
                zeroed = true;
            }
            // ---- S = Q K^T for this warp's 16 keys (two n8 tiles)
            float sfr[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int key = wk0 + (mi >> 1) * 8 + ri;
                const int ch = ks * 2 + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK + swz_off(key, ch), b0, b1, b2, b3);
                mma_bf16_16816(sfr[0], qa[ks], b0, b1);
                mma_bf16_16816(sfr[1], qa[ks], b2, b3);
            }
            // ---- mask, running max, probabilities
            float x[2][4];
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = wk0 + nt * 8 + 2 * qc + (e & 1);
                    const float v = key < nvalid ? sfr[nt][e] * c : -INFINITY;
                    x[nt][e] = v;
                    if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            // mn is finite: key wk0 (< nvalid) is unmasked in every row
            const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            uint32_t pa[4];
            float ps0 = 0.f, ps1 = 0.f, px0 = 0.f, px1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float e0 = ex2(x[nt][0] - mn0), e1 = ex2(x[nt][1] - mn0);
                const float e2 = ex2(x[nt][2] - mn1), e3 = ex2(x[nt][3] - mn1);
                const uint32_t lo = pack_bf16x2(e0, e1);
                const uint32_t hi = pack_bf16x2(e2, e3);
                ps0 += bf16lo_to_f32(lo) + bf16hi_to_f32(lo);
                ps1 += bf16lo_to_f32(hi) + bf16hi_to_f32(hi);
                px0 += e0 + e1;
                px1 += e2 + e3;
                pa[2 * nt] = lo;       // a0 / a2: row qr
                pa[2 * nt + 1] = hi;   // a1 / a3: row qr + 8
            }
            l0 = l0 * a0 + ps0;
            l1 = l1 * a1 + ps1;
            x0 = x0 * a0 + px0;
            x1 = x1 * a1 + px1;
            if (!__all_sync(0xFFFFFFFFu, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    oacc[i][0] *= a0;
                    oacc[i][1] *= a0;
                    oacc[i][2] *= a1;
                    oacc[i][3] *= a1;
                }
            }
            // ---- O += P V (V^T fragments via transposed ldmatrix)
#pragma unroll
            for (int pr = 0; pr < D / 16; ++pr) {
                const int key = wk0 + (mi & 1) * 8 + ri;
                const int ch = pr * 2 + (mi >> 1);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(sV + swz_off(key, ch), v0, v1, v2, v3);
                mma_bf16_16816(oacc[2 * pr], pa, v0, v1);
                mma_bf16_16816(oacc[2 * pr + 1], pa, v2, v3);
            }
        }
        if (zeroed) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
    }
    if (!ok) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        *abort_flag = 1;
    }
    // quad-reduce the per-thread partial sums
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    x0 += __shfl_xor_sync(0xFFFFFFFFu, x0, 1);
    x0 += __shfl_xor_sync(0xFFFFFFFFu, x0, 2);
    x1 += __shfl_xor_sync(0xFFFFFFFFu, x1, 1);
    x1 += __shfl_xor_sync(0xFFFFFFFFu, x1, 2);

    __syncthreads();  // ring drained (producer waited for its last copies)
    float* so = reinterpret_cast<float*>(smem + C::kScratchO);
    float* sm = reinterpret_cast<float*>(smem + C::kScratchM);
    float* sl = reinterpret_cast<float*>(smem + C::kScratchL);
    float* sx = reinterpret_cast<float*>(smem + C::kScratchX);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * qc;
        so[(warp * kMaxGroup + qr) * D + col] = oacc[i][0];
        so[(warp * kMaxGroup + qr) * D + col + 1] = oacc[i][1];
        so[(warp * kMaxGroup + qr + 8) * D + col] = oacc[i][2];
        so[(warp * kMaxGroup + qr + 8) * D + col + 1] = oacc[i][3];
    }
    if (qc == 0) {
        sm[warp * kMaxGroup + qr] = m0;
        sm[warp * kMaxGroup + qr + 8] = m1;
        sl[warp * kMaxGroup + qr] = l0;
        sl[warp * kMaxGroup + qr + 8] = l1;
        sx[warp * kMaxGroup + qr] = x0;
        sx[warp * kMaxGroup + qr + 8] = x1;
    }
    __syncthreads();
    const bool live = ok && !*abort_flag;
    const int tid = threadIdx.x;  // 0..127
    for (int e = tid; e < G * D && live; e += kConsumerWarps * 32) {
        const int h = e / D, col = e - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm[w * kMaxGroup + h]);
        float wsum = 0.f, xsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = sm[w * kMaxGroup + h];
            const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
            wsum += wt * sl[w * kMaxGroup + h];
            xsum += wt * sx[w * kMaxGroup + h];
            acc += wt * so[(w * kMaxGroup + h) * D + col];
        }
        const float val = acc / wsum;
        const float lse2 = M + log2f(xsum);
        const size_t bh = (size_t)b * p.Hq + (size_t)g * G + h;
        if (nsplit_b == 1) {
            if (col < p.dh) {
                if constexpr (OUT_F32) static_cast<float*>(o)[bh * p.dh + col] = val;
                else static_cast<__nv_bfloat16*>(o)[bh * p.dh + col] = __float2bfloat16_rn(val);
            }
            if (col == 0 && lse) lse[bh] = lse2 * kLn2f;
        } else {
            ws_o[(bh * p.max_splits + split) * D + col] = val;
            if (col == 0) ws_lse[bh * p.max_splits + split] = lse2;
        }
    }
    if (nsplit_b == 1 || p.slot < 0) return;
    // Count this split in (even after an abort, so that the count stays
    // whole); the CTA that completes the count merges the group.
    unsigned int* count = &g_dec_count[p.slot][kv_head];
    volatile int* is_last = abort_flag + 1;
    __threadfence();
    consumers_sync();
    if (tid == 0) *is_last = atomicAdd(count, 1u) == (unsigned int)(nsplit_b - 1);
    consumers_sync();
    if (!*is_last) return;
    __threadfence();
    // 1. the partials' LSEs of every (head, split) into shared memory, then per
    //    head (one warp each) M = max lse_s and the weights w_s = 2^(lse_s - M)
    // (the drained stage ring holds them: the host enables this merge only
    // when 2 * kMaxGroup + G * max_splits floats fit in it)
    float* s_head = reinterpret_cast<float*>(smem + C::kScratchO);  // [G][2]: 1/sum w, LSE
    float* s_w = s_head + 2 * kMaxGroup;                              // [G][nsplit_b]
    const size_t bh0 = (size_t)b * p.Hq + (size_t)g * G;
    for (int i = tid; i < G * nsplit_b; i += kConsumerWarps * 32) {
        const int h = i / nsplit_b, sp = i - h * nsplit_b;
        s_w[i] = __ldcg(ws_lse + (bh0 + h) * p.max_splits + sp);
    }
    consumers_sync();
    for (int h = warp; h < G; h += kConsumerWarps) {
        float M = -INFINITY;
        for (int sp = lane; sp < nsplit_b; sp += 32) M = fmaxf(M, s_w[h * nsplit_b + sp]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
        float sum = 0.f;
        for (int sp = lane; sp < nsplit_b; sp += 32) {
            const float w = ex2(s_w[h * nsplit_b + sp] - M);
            s_w[h * nsplit_b + sp] = w;
            sum += w;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        if (lane == 0) {
            s_head[2 * h] = 1.0f / sum;
            s_head[2 * h + 1] = (M + log2f(sum)) * kLn2f;
        }
    }
    consumers_sync();
    // 2. O = sum_s w_s o_s / sum_s w_s, four columns per thread, several
    //    splits' loads in flight
    for (int e = tid; e < G * (D / 4); e += kConsumerWarps * 32) {
        const int h = e / (D / 4), c4 = e - h * (D / 4);
        const float* wh = s_w + h * nsplit_b;
        const float4* src = reinterpret_cast<const float4*>(ws_o + (bh0 + h) * p.max_splits * D) + c4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int sp = 0; sp < nsplit_b; ++sp) {
            const float4 v = __ldcg(src + (size_t)sp * (D / 4));
            const float w = wh[sp];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        const float inv = s_head[2 * h];
        const size_t base = (bh0 + h) * p.dh + (size_t)c4 * 4;
        if (4 * c4 >= p.dh) {
            // a column group past the head dim: nothing to write
        } else if constexpr (OUT_F32) {
            *reinterpret_cast<float4*>(static_cast<float*>(o) + base) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + base) = pk;
        }
        if (c4 == 0 && lse) lse[bh0 + h] = s_head[2 * h + 1];
    }
    if (tid == 0) *count = 0u;
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(D)
attn_decode_combine_kernel(const int* __restrict__ seqlens, const float* __restrict__ ws_o,
                           const float* __restrict__ ws_lse, void* __restrict__ o,
                           float* __restrict__ lse, const DecParams p) {
    const int hq = blockIdx.x, b = blockIdx.y, col = threadIdx.x;
    int L = seqlens[b];
    L = L < 0 ? 0 : (L > p.Nmax ? p.Nmax : L);
    const int ns = (L + p.chunk - 1) / p.chunk;
    if (ns == 1) return;  // the split kernel wrote the final result
    const size_t bh = (size_t)b * p.Hq + hq;
    float val, lse_nat;
    if (ns == 0) {
        val = 0.f;
        lse_nat = -INFINITY;
    } else {
        const float* ls = ws_lse + bh * p.max_splits;
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s) M = fmaxf(M, ls[s]);
        float wsum = 0.f, acc = 0.f;
        for (int s = 0; s < ns; ++s) {
            const float w = ex2(ls[s] - M);
            wsum += w;
            acc += w * ws_o[(bh * p.max_splits + s) * D + col];
        }
        val = acc / wsum;
        lse_nat = (M + log2f(wsum)) * kLn2f;
    }
    if (col < p.dh) {
        if constexpr (OUT_F32) static_cast<float*>(o)[bh * p.dh + col] = val;
        else static_cast<__nv_bfloat16*>(o)[bh * p.dh + col] = __float2bfloat16_rn(val);
    }
    if (col == 0 && lse) lse[bh] = lse_nat;
}

template <int D, bool OUT_F32>
attn_status_t launch_decode_t(const CUtensorMap& tk, const CUtensorMap& tv, const void* q,
                              const int* seqlens, void* o, float* lse, float* ws_o, float* ws_lse,
                              const DecParams& p, cudaStream_t stream, const DeviceInfo& dev) {
    using C = DecCfg<D>;
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_decode_split_kernel<D, OUT_F32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    const DecParams& pk = p;
    dim3 grid((unsigned)p.max_splits, (unsigned)p.Hkv, (unsigned)p.B);
    attn_decode_split_kernel<D, OUT_F32><<<grid, kDecThreads, C::kSmemBytes, stream>>>(
        tk, tv, static_cast<const __nv_bfloat16*>(q), seqlens, o, lse, ws_o, ws_lse, pk,
        dev.err_word);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (pk.slot >= 0) return ATTN_OK;  // merged in the split kernel
    dim3 cgrid((unsigned)p.Hq, (unsigned)p.B);
    attn_decode_combine_kernel<D, OUT_F32><<<cgrid, D, 0, stream>>>(seqlens, ws_o, ws_lse, o, lse, pk);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

bool decode_merges_in_kernel(int B, int Hkv, int G, int max_splits, int d) {
    // counter table, and the split weights in the drained stage ring
    const size_t ring_floats =
        (size_t)(d == 256 ? DecCfg<256>::kBarOff : d == 128 ? DecCfg<128>::kBarOff : DecCfg<64>::kBarOff) / 4;
    return (long long)B * Hkv <= kDecMaxGroups &&
           (size_t)(2 * kMaxGroup) + (size_t)G * (size_t)max_splits <= ring_floats;
}

int decode_chunk(int Nmax, int B, int Hkv, int num_sms, int num_splits) {
    int s = num_splits;
    const int max_tiles = (Nmax + kStageKeys - 1) / kStageKeys;
    if (s <= 0) {
        s = attn_decode_num_splits(B * Hkv, num_sms, max_tiles < 128 ? max_tiles : 128);
        if (s <= 0) s = 1;
    }
    int chunk = (Nmax + s - 1) / s;
    chunk = (chunk + kStageKeys - 1) / kStageKeys * kStageKeys;
    if (num_splits <= 0 && chunk > kAutoMaxChunk) chunk = kAutoMaxChunk;
    if (chunk < kStageKeys) chunk = kStageKeys;
    return chunk;
}

static size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

size_t decode_workspace_bytes(int B, int Hq, int Nmax, int d, int chunk) {
    const size_t max_splits = (size_t)((Nmax + chunk - 1) / chunk);
    const size_t rows = (size_t)B * Hq * max_splits;
    return align16(rows * d * 4) + align16(rows * 4);
}

namespace {
attn_status_t launch_decode_common(const CUtensorMap& tk, const CUtensorMap& tv, const void* q,
                                   const int* seqlens, void* o, float* lse, DecParams& p, int d,
                                   void* workspace, attn_out_dtype_t o_dtype, cudaStream_t stream,
                                   const DeviceInfo& dev) {
    d = decode_pad_head_dim(d);  // the kernel's tile width (columns past p.dh are zeros)
    const size_t rows = (size_t)p.B * p.Hq * p.max_splits;
    float* ws_o = static_cast<float*>(workspace);
    float* ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align16(rows * d * 4));
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if (d == 256)
        return f32 ? launch_decode_t<256, true>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev)
                   : launch_decode_t<256, false>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev);
    if (d == 128)
        return f32 ? launch_decode_t<128, true>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev)
                   : launch_decode_t<128, false>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev);
    if (d == 64)
        return f32 ? launch_decode_t<64, true>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev)
                   : launch_decode_t<64, false>(tk, tv, q, seqlens, o, lse, ws_o, ws_lse, p, stream, dev);
    return ATTN_ERR_UNSUPPORTED;  // d is the padded head dim here
}

DecParams make_dec_params(int B, int Hq, int Hkv, int Nmax, int d, float scale, int chunk) {
    DecParams p;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Nmax = Nmax;
    p.chunk = chunk;
    p.max_splits = (Nmax + chunk - 1) / chunk;
    p.c = scale * kLog2ef;
    static std::atomic<uint32_t> launches{0};
    p.slot = decode_merges_in_kernel(B, Hkv, p.G, p.max_splits, decode_pad_head_dim(d))
                 ? (int)(launches.fetch_add(1u, std::memory_order_relaxed) % kDecSlots)
                 : -1;
    p.block_table = nullptr;
    p.page_size = 0;
    p.max_blocks = 0;
    p.dh = d;
    return p;
}
}  // namespace

attn_status_t launch_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                            int Nmax, int d, float scale, int chunk, void* workspace,
                            attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev) {
    DecParams p = make_dec_params(B, Hq, Hkv, Nmax, d, scale, chunk);
    CUtensorMap tk, tv;
    attn_status_t st;
    if ((st = encode_tmap_bf16_3d(&tk, k_cache, d, Nmax, (long long)B * Hkv, kStageKeys)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tv, v_cache, d, Nmax, (long long)B * Hkv, kStageKeys)) != ATTN_OK) return st;
    return launch_decode_common(tk, tv, q, seqlens, o, lse, p, d, workspace, o_dtype, stream, dev);
}

attn_status_t launch_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                  const int* block_table, const int* seqlens, void* o, float* lse,
                                  int B, int Hq, int Hkv, long long num_blocks, int page_size,
                                  int max_blocks, int d, float scale, int chunk, void* workspace,
                                  attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev) {
    const int Nmax = max_blocks * page_size;
    DecParams p = make_dec_params(B, Hq, Hkv, Nmax, d, scale, chunk);
    p.block_table = block_table;
    p.page_size = page_size;
    p.max_blocks = max_blocks;
    CUtensorMap tk, tv;
    attn_status_t st;
    if ((st = encode_tmap_paged_kv(&tk, k_pages, d, Hkv, page_size, num_blocks)) != ATTN_OK) return st;
    if ((st = encode_tmap_paged_kv(&tv, v_pages, d, Hkv, page_size, num_blocks)) != ATTN_OK) return st;
    return launch_decode_common(tk, tv, q, seqlens, o, lse, p, d, workspace, o_dtype, stream, dev);
}

}  // namespace gb300

// ---------------------------------------------------------------------------
// attn_decode_noalloc: the same decode with a scratch buffer the library owns.
//
// Some callers cannot call cudaMalloc at all -- for example a plugin inside a
// host framework that hands all device memory to its own pool and offers no
// allocator, or a latency-critical loop where an allocation's implicit device
// synchronisation is not acceptable.  For them the split partials live in one
// fixed array in device global memory, reserved when the library is loaded on
// a GPU and held until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace gb300 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of g_decode_scratch on the current device.  Host code must
// not pass the symbol itself to a kernel (on the host it is only a stand-in),
// so the address is looked up once per device, with that device current.
attn_status_t scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}
}  // namespace

}  // namespace gb300

extern "C" attn_status_t attn_decode_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int* seqlens, void* o,
                                             float* lse, int B, int Hq, int Hkv, int Nmax, int d,
                                             float scale, int num_splits,
                                             attn_out_dtype_t o_dtype, void* stream) {
    // attn_decode's own argument checks first, so both entry points reject a
    // bad call with the same status
    const attn_status_t chk = gb300::check_decode_call(q, k_cache, v_cache, seqlens, o, lse, B, Hq,
                                                       Hkv, Nmax, d, scale, num_splits, o_dtype);
    if (chk != ATTN_OK) return chk;
    const size_t need = attn_decode_workspace_size(B, Hq, Hkv, Nmax, d, num_splits);
    if (need == 0)  // no usable device: let attn_decode report it
        return attn_decode(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Nmax, d, scale,
                           num_splits, nullptr, 0, o_dtype, stream);
    if (need > gb300::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
    void* ws = nullptr;
    const attn_status_t st = gb300::scratch_address(&ws);
    if (st != ATTN_OK) return st;
    return attn_decode(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Nmax, d, scale,
                       num_splits, ws, gb300::kNoAllocScratchBytes, o_dtype, stream);
}
