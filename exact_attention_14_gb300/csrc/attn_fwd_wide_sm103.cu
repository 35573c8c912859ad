// attn_fwd_wide_sm103.cu -- fused attention forward for head dims above 128
// (d in (128, 256], run on kernels built for D = 192 and D = 256).
//
// The 128-column forward keeps two 128-row Q tiles in flight per CTA, each with
// a 128-column S and a d-column O in tensor memory; at d > 128 two O
// accumulators no longer fit next to their S tiles in the 512 TMEM columns.
// This kernel keeps one Q tile per CTA and overlaps the other way: two S
// buffers of 128 keys, so S(j+1) is computed while the softmax warps work on
// S(j) (TMEM: O [0, D), S0 [256, 384), S1 [384, 512)).  Per 128-key tile the
// tensor cores do 2 * 128 * 128 * D * 2 FLOPs, which at D = 256 outweighs the
// softmax work of the tile; with N = 128 keys the S product reads its operands
// from shared memory at the tensor cores' full rate (N = 64 would not).
// K and V reach shared memory through one ring of 32 KiB slots, filled in the
// order the MMAs consume them: K_j as two column chunks (d 0-127 and 128-D,
// 128 keys each) and V_j as two 64-key halves.  A K/V tile pair of 128 keys at
// D = 256 is 128 KiB, so whole tiles could not be double-buffered next to Q.
//
// Roles (8 warps): warp 0 TMA producer (Q once per unit, K and V chunks
// through the ring), warp 1 MMA issuer and TMEM owner, warps 2-3 idle,
// warps 4-7 softmax (one query row per thread) and epilogue.  Persistent CTAs
// take units (b, query head, 128-row Q tile) from a device-side queue in the
// order of fwd_sched.h (L2 sections; causal longest-first).
//
// MMA order per unit of n tiles: S(0), S(1), then for each tile j once P(j) is
// in TMEM: PV(j), S(j + 2) into the buffer PV(j) has read (one CTA's MMAs run
// in issue order).  Because S(j + 1) may finish before PV(j - 1), the softmax
// rescales O (lecture notes 5.3, tau = 8) only after waiting for the P.V
// product of the previous tile (a barrier committed after every PV).
//
// Method: lecture notes "Optimizing Attention for Modern Hardware:
// FlashAttention 1-4", 2.2 online softmax, 2.5 causal block skipping, 2.6 / 3.2
// delayed normalisation and the logsumexp, 4.5 persistent kernel, 5.3
// conditional rescaling; the head dims the pages list for the FlashAttention
// kernels (64, 96, 128, 192, 256) and their warning about other head dims
// ("FlashAttention: tiling + recomputation", 6, pitfall 1).
#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "fwd_sched.h"

namespace gb300 {
namespace {

constexpr int kWThreads = 256;
constexpr int kWM = 128;   // query rows per Q tile
constexpr int kWN = 128;   // keys per K/V tile (and S buffer)
constexpr int kWV = 64;    // keys per V chunk
constexpr int kWSlots = 5;                // ring slots
constexpr int kWSlotBytes = 32768;
constexpr float kWTau = 8.0f;
constexpr float kWLn2 = 0.69314718055994530942f;
constexpr float kWLog2e = 1.44269504088896340736f;
constexpr uint32_t kWNegInf = 0xFF800000u;

template <int D>
struct WideCfg {
    static constexpr int kQBytes = kWM * D * 2;     // D / 64 chunks of 128 rows x 128 B
    // ring entries: K chunk c (128 keys x columns [128 c, min(128 c + 128, D)),
    // 64-column pieces of 128 rows x 128 B) and V half h (64 keys x D, 64-column
    // pieces of 64 rows x 128 B)
    static __host__ __device__ constexpr int kKChunkBytes(int c) { return kWN * (D - 128 * c < 128 ? D - 128 * c : 128) * 2; }
    static constexpr int kVHalfBytes = kWV * D * 2;
    static constexpr int kRing = kQBytes;
    static constexpr int kBar = kRing + kWSlots * kWSlotBytes;
    static constexpr int kSmemBytes = kBar + 512 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kKChunkBytes(0) <= kWSlotBytes && kKChunkBytes(1) <= kWSlotBytes &&
                  kVHalfBytes <= kWSlotBytes, "ring slot size");
    static_assert(D > 128 && D <= 256, "two K column chunks");
    static constexpr uint32_t kColO = 0;
    static __host__ __device__ constexpr uint32_t col_s(int b) { return 256u + 128u * (uint32_t)b; }
};

__host__ __device__ constexpr int wide_epi_cols(bool f32) { return f32 ? 16 : 32; }

struct WideParams {
    FwdShape shape;   // nmb counts 128-row Q tiles here
    int group, off, d_act;
    float c;          // scale * log2(e)
    uint32_t slot;
    void* o;          // O: [B, Hq, Nq, d_act], or [total_q, Hq, d_act] for packed batches
    // packed batches: Nq / Nk in shape are the longest sequence's lengths
    const int* cu_q;  // [B + 1] row offsets in the packed Q / O
    const int* cu_k;  // [B + 1] row offsets in the packed K / V
    int total_q, total_k;
};

constexpr uint32_t kWideQueueSlots = 256;
__device__ unsigned int g_wide_queue[kWideQueueSlots][2];  // ticket counter, exit count

struct WItem {
    int bh, mt, n;
    int q0, nq, nk;  // packed batches: the sequence's first row and lengths
};

struct __align__(8) WideBars {
    uint64_t q_full, q_empty;
    uint64_t ring_full[kWSlots], ring_empty[kWSlots];
    uint64_t s_full[2], p_full[2], pv_done, o_full;
    uint64_t unit_full[2], unit_empty[2];
    uint64_t drain;
    WItem item[2];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(WideBars) <= 512, "barrier block");

constexpr int kWConsumers = 5;  // MMA warp + 4 softmax warps

// KV tiles of 128 keys that Q tile mt (rows [128 mt, 128 mt + 128)) needs.
__device__ __forceinline__ int wide_kv_tiles(const FwdShape& s, int mt) {
    const int r0 = mt * kWM;
    int rows = s.Nq - r0;
    rows = rows < kWM ? rows : kWM;
    return kv_tiles_for_rows(r0, rows, s.Nq, s.Nk, s.causal, kWN);
}

__device__ __forceinline__ bool take_witem(WideBars* bars, uint32_t k, WItem& w,
                                           const volatile int* abort_flag) {
    const uint32_t i = k & 1u;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_full[i]), (k >> 1) & 1u, abort_flag)))
        return false;
    const volatile WItem* src = &bars->item[i];
    w.bh = src->bh;
    w.mt = src->mt;
    w.n = src->n;
    w.q0 = src->q0;
    w.nq = src->nq;
    w.nk = src->nk;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars->unit_empty[i]));
    return true;
}

__device__ __forceinline__ void wide_abort(WideBars* bars, unsigned int* err) {
    atomicOr(err, kErrTimeout);
    *((volatile int*)&bars->abort) = 1;
}

// Sequence b of a packed batch: its first rows and lengths (the checks of the
// 128-column forward's packed path).  False, and the error bit from the
// leader, when its offsets leave the arrays, decrease, or give a length above
// the launch's maximum, a query row without keys, or, causal, more queries
// than keys; such a sequence is not computed.
__device__ __forceinline__ bool wide_varlen_seq(const WideParams& p, int b, bool leader, int& q0,
                                                int& nq, int& k0, int& nk, unsigned int* err) {
    const int qs = __ldg(p.cu_q + b), qe = __ldg(p.cu_q + b + 1);
    const int ks = __ldg(p.cu_k + b), ke = __ldg(p.cu_k + b + 1);
    const bool good = 0 <= qs && qs <= qe && qe <= p.total_q && qe - qs <= p.shape.Nq &&
                      0 <= ks && ks <= ke && ke <= p.total_k && ke - ks <= p.shape.Nk &&
                      (qe == qs || ke > ks) && (!p.shape.causal || qe - qs <= ke - ks);
    q0 = qs; nq = qe - qs; k0 = ks; nk = ke - ks;
    if (!good && leader) atomicOr(err, kErrBadSeqlen);
    return good;
}

template <int D, bool VARLEN>
__device__ void wide_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              uint8_t* smem, WideBars* bars, const WideParams& p, unsigned int* err) {
    using C = WideCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1;
    unsigned int* queue = g_wide_queue[p.slot];
    int q_loads = 0;    // Q loads issued
    long long L = 0;    // ring entries issued
    bool ok = true;
    for (int local = 0; ok; ++local) {
        const uint32_t hs = (uint32_t)local & 1u;
        if (local >= 2)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_empty[hs]),
                                                   (uint32_t)((local >> 1) - 1) & 1u, abort_flag));
        if (!ok) break;
        // A CTA's first unit is its own index, later ones come from the
        // counter; packed batches skip the units past their sequence's end.
        bool done = false;
        int bh = -1, mt = 0, n = 0;
        int q0 = 0, k0 = 0, nq = s.Nq, nk = s.Nk;
        while (true) {
            uint32_t u = blockIdx.x;
            if (local > 0 || (VARLEN && bh >= 0)) {
                if (leader) u = gridDim.x + atomicAdd(&queue[0], 1u);
                u = __shfl_sync(0xFFFFFFFFu, u, leader_lane);
            }
            done = u >= (uint32_t)s.units;
            if (done) {
                bh = -1;
                break;
            }
            unit_of(s, u, bh, mt);
            if constexpr (VARLEN) {
                if (!wide_varlen_seq(p, bh / s.Hq, leader, q0, nq, k0, nk, err)) continue;
                if (mt * kWM >= nq) continue;
            }
            break;
        }
        if (!done) {
            if constexpr (VARLEN) {
                const int r0 = mt * kWM;
                n = kv_tiles_for_rows(r0, nq - r0 < kWM ? nq - r0 : kWM, nq, nk, s.causal, kWN);
            } else {
                n = wide_kv_tiles(s, mt);
            }
        }
        if (leader) {
            volatile WItem* dst = &bars->item[hs];
            dst->bh = bh;
            dst->mt = mt;
            dst->n = n;
            dst->q0 = q0;
            dst->nq = nq;
            dst->nk = nk;
            mbar_arrive(smem_u32(&bars->unit_full[hs]));
        }
        __syncwarp();
        if (done) break;
        const int b = bh / s.Hq;
        const int hq = bh - b * s.Hq;
        // the K/V head: an index into [B * Hkv] dense, into [Hkv] packed
        const int kvh = VARLEN ? hq / p.group : b * s.Hkv + hq / p.group;
        if (q_loads > 0)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->q_empty), (uint32_t)(q_loads - 1) & 1u,
                                                   abort_flag));
        if (!ok) break;
        if (leader) {
            const uint32_t bar = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(bar, C::kQBytes);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                if constexpr (VARLEN)
                    tma_load_5d(smem_u32(smem) + c * (kWM * 128), tq, bar, 64 * c, hq,
                                kRaggedWindow - nq + mt * kWM, q0 + nq, kRaggedWindow);
                else
                    tma_load_3d(smem_u32(smem) + c * (kWM * 128), tq, bar, 64 * c, mt * kWM, bh);
            }
        }
        __syncwarp();
        ++q_loads;
        // ring entries in the MMA warp's order: K_0, K_1, then per tile j
        // V_j and K_{j+2}
        auto emit_k = [&](int j) {
            for (int c = 0; c < 2 && ok; ++c) {
                const int slot = (int)(L % kWSlots);
                if (L >= kWSlots)
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->ring_empty[slot]),
                                                           (uint32_t)((L / kWSlots - 1) & 1), abort_flag));
                if (!ok) return;
                if (leader) {
                    const uint32_t bar = smem_u32(&bars->ring_full[slot]);
                    mbar_arrive_expect_tx(bar, C::kKChunkBytes(c));
                    const uint32_t dst = smem_u32(smem + C::kRing + slot * kWSlotBytes);
                    const int pieces = C::kKChunkBytes(c) / (kWN * 128);
                    for (int pc = 0; pc < pieces; ++pc) {
                        if constexpr (VARLEN)
                            tma_load_5d(dst + pc * (kWN * 128), tk, bar, 128 * c + 64 * pc, kvh,
                                        kRaggedWindow - nk + j * kWN, k0 + nk, kRaggedWindow);
                        else
                            tma_load_3d(dst + pc * (kWN * 128), tk, bar, 128 * c + 64 * pc, j * kWN, kvh);
                    }
                }
                __syncwarp();
                ++L;
            }
        };
        auto emit_v = [&](int j) {
            for (int h = 0; h < 2 && ok; ++h) {
                const int slot = (int)(L % kWSlots);
                if (L >= kWSlots)
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->ring_empty[slot]),
                                                           (uint32_t)((L / kWSlots - 1) & 1), abort_flag));
                if (!ok) return;
                if (leader) {
                    const uint32_t bar = smem_u32(&bars->ring_full[slot]);
                    mbar_arrive_expect_tx(bar, C::kVHalfBytes);
                    const uint32_t dst = smem_u32(smem + C::kRing + slot * kWSlotBytes);
#pragma unroll
                    for (int pc = 0; pc < D / 64; ++pc) {
                        if constexpr (VARLEN)
                            tma_load_5d(dst + pc * (kWV * 128), tv, bar, 64 * pc, kvh,
                                        kRaggedWindow - nk + j * kWN + kWV * h, k0 + nk, kRaggedWindow);
                        else
                            tma_load_3d(dst + pc * (kWV * 128), tv, bar, 64 * pc, j * kWN + kWV * h, kvh);
                    }
                }
                __syncwarp();
                ++L;
            }
        };
        emit_k(0);
        if (n > 1) emit_k(1);
        for (int j = 0; j < n && ok; ++j) {
            emit_v(j);
            if (j + 2 < n) emit_k(j + 2);
        }
    }
    if (!ok && leader) wide_abort(bars, err);
    if (leader) {
        __threadfence();
        if (atomicAdd(&queue[1], 1u) == gridDim.x - 1) {
            queue[0] = 0u;
            queue[1] = 0u;
        }
    }
    // Drain: every issued copy lands before the CTA may exit.
    if (q_loads > 0) mbar_wait(smem_u32(&bars->q_full), (uint32_t)(q_loads - 1) & 1u, nullptr);
    for (int st = 0; st < kWSlots && st < L; ++st) {
        const long long uses = (L - st + kWSlots - 1) / kWSlots;
        mbar_wait(smem_u32(&bars->ring_full[st]), (uint32_t)((uses - 1) & 1), nullptr);
    }
    __syncwarp();
}

constexpr uint32_t kWDescHi = sdesc_hi_sw128(1024);

// S = Q K_j^T, k-steps [kk0, kk1) of 16 columns: M = 128, N = 128.  Q is
// D / 64 pieces of 128 rows x 128 B (16 KiB apart); the K chunk holding
// columns [128 c, 128 c + 128) is two such pieces of its own.
template <int D>
__device__ __forceinline__ void wide_issue_s(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo, int kk0,
                                             int kk1, uint32_t idesc) {
#pragma unroll
    for (int kk = kk0; kk < kk1; ++kk) {
        const uint32_t in = (kk & 3) * (32 >> 4);
        mma_ss_warp(d_tmem, sdesc_join(q_lo + (kk >> 2) * ((kWM * 128) >> 4) + in, kWDescHi),
                    sdesc_join(k_lo + ((kk >> 2) & 1) * ((kWN * 128) >> 4) + in, kWDescHi), idesc,
                    kk > 0 ? 1u : 0u);
    }
}

// O += P V for one 64-key half of V_j: A = P (bf16 pairs in TMEM, 8 columns
// per 16 keys), B = the half MN-major (LBO 8 KiB between 64-column pieces,
// 16 keys = 16 rows of 128 B).
__device__ __forceinline__ void wide_issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                              uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kWV / 16; ++kk)
        mma_ts_warp(d_tmem, p_tmem + kk * 8, sdesc_join(v_lo + kk * (2048 >> 4), kWDescHi), idesc,
                    (accumulate || kk > 0) ? 1u : 0u);
}

template <int D>
__device__ void wide_mma(uint8_t* smem, WideBars* bars, uint32_t tmem, unsigned int* err) {
    using C = WideCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idS = make_idesc_bf16(kWM, kWN, 0, 0);
    const uint32_t idO = make_idesc_bf16(kWM, D, 0, 1);
    const uint32_t q_lo = sdesc_lo(smem_u32(smem), 16);
    auto k_lo = [&](int st) { return sdesc_lo(smem_u32(smem + C::kRing + st * kWSlotBytes), 16); };
    auto v_lo = [&](int st) {
        return sdesc_lo(smem_u32(smem + C::kRing + st * kWSlotBytes), kWV * 128);
    };
    auto wait_all = [&](uint32_t bar, uint32_t parity, int polls) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, polls));
    };
    long long g = 0;   // tiles of all units so far: tile g uses S buffer g & 1
    long long L = 0;   // ring entries consumed
    bool ok = true;
    // The next ring entry, once it has landed.
    auto take = [&](int& slot) {
        slot = (int)(L % kWSlots);
        if (!wait_all(smem_u32(&bars->ring_full[slot]), (uint32_t)((L / kWSlots) & 1), 0)) return false;
        tc_fence_after();
        ++L;
        return true;
    };
    // S for global tile gg into buffer gg & 1 (K_j's two column chunks).
    auto issue_s = [&](long long gg, bool last_s) {
        const uint32_t dS = tmem + C::col_s((int)(gg & 1));
        int slot;
        if (!take(slot)) return false;
        wide_issue_s<D>(dS, q_lo, k_lo(slot), 0, 8, idS);
        mma_commit_warp(smem_u32(&bars->ring_empty[slot]));
        if (!take(slot)) return false;
        wide_issue_s<D>(dS, q_lo, k_lo(slot), 8, D / 16, idS);
        mma_commit_warp(smem_u32(&bars->ring_empty[slot]));
        mma_commit_warp(smem_u32(&bars->s_full[gg & 1]));
        if (last_s) mma_commit_warp(smem_u32(&bars->q_empty));
        return true;
    };
    for (int local = 0; ok; ++local) {
        WItem w;
        ok = take_witem(bars, (uint32_t)local, w, abort_flag);
        if (!ok || w.bh < 0) break;
        const int n = w.n;
        ok = wait_all(smem_u32(&bars->q_full), (uint32_t)local & 1u, 0);
        if (!ok) break;
        ok = issue_s(g, n == 1);
        if (ok && n > 1) ok = issue_s(g + 1, n == 2);
        for (int j = 0; j < n && ok; ++j, ++g) {
            const int b = (int)(g & 1);
            ok = wait_all(smem_u32(&bars->p_full[b]), (uint32_t)((g >> 1) & 1), 32);
            if (!ok) break;
            for (int h = 0; h < 2 && ok; ++h) {
                int slot;
                ok = take(slot);
                if (!ok) break;
                wide_issue_pv(tmem + C::kColO, tmem + C::col_s(b) + (uint32_t)(h * 32), v_lo(slot), idO,
                              j > 0 || h > 0);
                mma_commit_warp(smem_u32(&bars->ring_empty[slot]));
            }
            if (!ok) break;
            mma_commit_warp(smem_u32(&bars->pv_done));
            if (j + 2 < n) {
                ok = issue_s(g + 2, j + 3 == n);
                if (!ok) break;
            }
            if (j + 1 == n) mma_commit_warp(smem_u32(&bars->o_full));
        }
    }
    if (!ok && leader) wide_abort(bars, err);
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// One 128-key tile of the online softmax for this thread's row (see the 128-
// column forward): mask, tile max, conditional rescale of O (after the
// previous P.V product has completed), P = 2^(s c - m) to TMEM as bf16 pairs,
// and the two row sums.
template <int D, bool MASKED>
__device__ __forceinline__ void wide_softmax_tile(uint32_t (&sr)[kWN], int lim, bool first, float c,
                                                  uint32_t tP, uint32_t tO, float& m, float& l,
                                                  float& lx, WideBars* bars, long long g,
                                                  const volatile int* abort_flag, bool& ok) {
    if constexpr (MASKED) {
#pragma unroll
        for (int cc = 0; cc < kWN; ++cc)
            if (cc > lim) sr[cc] = kWNegInf;
    }
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < kWN; cc += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[cc + 4]), __uint_as_float(sr[cc + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[cc + 6]), __uint_as_float(sr[cc + 7]));
    }
    const float smax = fmax3(fmaxf(mx0, mx1), mx2, mx3);
    const float mt = smax * c;
    const bool need = mt > m + kWTau;
    if (__any_sync(0xFFFFFFFFu, need)) {
        const float m_new = fmaxf(m, mt);
        const float alpha = ex2(m - m_new);
        l *= alpha;
        lx *= alpha;
        if (!first) {
            // O must hold the previous tile's product before it is rescaled
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->pv_done), (uint32_t)((g - 1) & 1),
                                                   abort_flag));
            if (!ok) return;
            tc_fence_after();
            const uint64_t a2 = f2(alpha, alpha);
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t r[32];
                tmem_ld32(tO + cc, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float lo, hi;
                    f2_split(f2_mul(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), a2), lo, hi);
                    r[i] = __float_as_uint(lo);
                    r[i + 1] = __float_as_uint(hi);
                }
                tmem_st32(tO + cc, r);
            }
        }
        m = m_new;
    }
    {
        const float pmax = ex2(fmaf(smax, c, -m));
        l += bf16lo_to_f32(pack_bf16x2(pmax, 0.f)) - pmax;
    }
    const uint64_t c2 = f2(c, c), nm2 = f2(-m, -m);
    uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
    for (int half = 0; half < kWN / 32; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int col = half * 32 + 2 * i;
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), c2, nm2), x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if constexpr (MASKED) {
                p0 = col <= lim ? p0 : 0.f;
                p1 = col + 1 <= lim ? p1 : 0.f;
            }
            pk[i] = pack_bf16x2(p0, p1);
            if (i & 1)
                acc1 = f2_add(acc1, f2(p0, p1));
            else
                acc0 = f2_add(acc0, f2(p0, p1));
        }
        tmem_st16(tP + half * 16, pk);
    }
    float a, bb;
    f2_split(f2_add(acc0, acc1), a, bb);
    lx += a + bb;
    l += a + bb;
}

// Epilogue store of 32 columns [cc, cc + 32) of this warp's 32 rows of O
// straight from registers, whole 32-byte sectors per store: lanes 2k and 2k+1
// swap one 16-byte piece of each sector, then both write row 2k's sector and,
// in the next store, row 2k+1's (no shared memory, which the S MMAs' operand
// reads keep busy).  Run by the whole warp; rows at or past rows_live and
// 16-byte pieces at or past d_act (a multiple of 8) are not written.
template <bool OUT_F32>
__device__ __forceinline__ void wide_store_pairs(const float (&v)[32], int cc, int lane, uint8_t* o_warp,
                                                 size_t row_stride, int rows_live, int d_act) {
    constexpr int kEs = OUT_F32 ? 4 : 2;
    constexpr int kPieces = 32 * kEs / 16;
    constexpr int kColsPerPiece = 16 / kEs;
    uint32_t wd[kPieces * 4];
    if constexpr (OUT_F32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) wd[i] = __float_as_uint(v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) wd[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
    const bool odd = lane & 1;
    const int ra = lane & ~1, rb = lane | 1;
    uint8_t* pa = o_warp + (size_t)ra * row_stride + (size_t)cc * kEs + (odd ? 16 : 0);
    uint8_t* pb = o_warp + (size_t)rb * row_stride + (size_t)cc * kEs + (odd ? 16 : 0);
    const bool live_a = ra < rows_live, live_b = rb < rows_live;
#pragma unroll
    for (int sct = 0; sct < kPieces / 2; ++sct) {
        if (cc + 2 * sct * kColsPerPiece >= d_act) break;
        const int pe = 2 * sct, po = 2 * sct + 1;
        const bool col_ok = cc + (odd ? po : pe) * kColsPerPiece < d_act;
        uint32_t da[4], db[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t x = odd ? wd[pe * 4 + i] : wd[po * 4 + i];
            const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
            da[i] = odd ? y : wd[pe * 4 + i];
            db[i] = odd ? wd[po * 4 + i] : y;
        }
        if (live_a && col_ok) *reinterpret_cast<uint4*>(pa + sct * 32) = make_uint4(da[0], da[1], da[2], da[3]);
        if (live_b && col_ok) *reinterpret_cast<uint4*>(pb + sct * 32) = make_uint4(db[0], db[1], db[2], db[3]);
    }
}

template <int D, bool OUT_F32, bool VARLEN>
__device__ void wide_softmax(int wq, int lane, uint8_t* smem, WideBars* bars, uint32_t tmem,
                             const WideParams& p, const CUtensorMap* to, float* __restrict__ lse_ptr,
                             unsigned int* err) {
    using C = WideCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tO = tmem + C::kColO + lane_off;
    long long g = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
        WItem w;
        ok = take_witem(bars, k, w, abort_flag);
        if (!ok || w.bh < 0) break;
        const int row = w.mt * kWM + wq * 32 + lane;
        const int nq = VARLEN ? w.nq : s.Nq;
        const int nk = VARLEN ? w.nk : s.Nk;
        int last_key = nk - 1;
        if (s.causal) {
            const int lk = row + (VARLEN ? nk - nq : p.off);
            last_key = lk < last_key ? lk : last_key;
        }
        float m = -INFINITY, l = 0.f, lx = 0.f;
        for (int j = 0; j < w.n && ok; ++j, ++g) {
            const int b = (int)(g & 1);
            const uint32_t tS = tmem + C::col_s(b) + lane_off;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->s_full[b]), (uint32_t)((g >> 1) & 1),
                                                   abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[kWN];
#pragma unroll
            for (int cc = 0; cc < kWN; cc += 32)
                tmem_ld32(tS + cc, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc]));
            tmem_wait_ld();
            const int lim = last_key - j * kWN;
            if (__any_sync(0xFFFFFFFFu, lim < kWN - 1))
                wide_softmax_tile<D, true>(sr, lim, j == 0, p.c, tS, tO, m, l, lx, bars, g, abort_flag, ok);
            else
                wide_softmax_tile<D, false>(sr, lim, j == 0, p.c, tS, tO, m, l, lx, bars, g, abort_flag, ok);
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[b]));
        }
        if (!ok) break;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->o_full), k & 1u, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const uint64_t il2 = f2(inv_l, inv_l);
        const int row0 = w.mt * kWM + wq * 32;
        constexpr int kEs = OUT_F32 ? 4 : 2;
        const int hq = w.bh - (w.bh / s.Hq) * s.Hq;
        // this warp's first row of O and the stride between rows
        const size_t first = VARLEN ? (size_t)(w.q0 + row0) * s.Hq + (size_t)hq
                                    : (size_t)w.bh * s.Nq + (size_t)row0;
        const size_t row_stride = (VARLEN ? (size_t)s.Hq : 1u) * (size_t)p.d_act * kEs;
        uint8_t* o_warp = static_cast<uint8_t*>(p.o) + first * p.d_act * kEs;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
            uint32_t r[32];
            tmem_ld32(tO + cc, r);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2)
                f2_split(f2_mul(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), il2), v[i], v[i + 1]);
            wide_store_pairs<OUT_F32>(v, cc, lane, o_warp, row_stride, nq - row0, p.d_act);
        }
        // LSE: [B, Hq, Nq], or [Hq, total_q] for packed batches
        if (row < nq && lse_ptr)
            lse_ptr[VARLEN ? (size_t)hq * p.total_q + (size_t)(w.q0 + row)
                           : (size_t)w.bh * s.Nq + (size_t)row] = (m + log2f(lx)) * kWLn2;
        // (the next unit's P.V overwrites O only after this warpgroup's next
        // P is in TMEM, which follows these loads)
    }
    if (!ok) wide_abort(bars, err);
}

template <int D, bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kWThreads, 1)
attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                     float* __restrict__ lse_ptr, const WideParams p, unsigned int* err) {
    using C = WideCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    WideBars* bars = reinterpret_cast<WideBars*>(smem + C::kBar);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_empty), 1);
        for (int i = 0; i < kWSlots; ++i) {
            mbar_init(smem_u32(&bars->ring_full[i]), 1);
            mbar_init(smem_u32(&bars->ring_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->s_full[i]), 1);
            mbar_init(smem_u32(&bars->p_full[i]), 4);
            mbar_init(smem_u32(&bars->unit_full[i]), 1);
            mbar_init(smem_u32(&bars->unit_empty[i]), kWConsumers);
        }
        mbar_init(smem_u32(&bars->pv_done), 1);
        mbar_init(smem_u32(&bars->o_full), 1);
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
    if (warp == 0) wide_producer<D, VARLEN>(&tq, &tk, &tv, smem, bars, p, err);
    else if (warp == 1) wide_mma<D>(smem, bars, tmem, err);
    else if (warp >= 4)
        wide_softmax<D, OUT_F32, VARLEN>(warp & 3, lane, smem, bars, tmem, p, &to, lse_ptr, err);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool OUT_F32, bool VARLEN = false>
attn_status_t launch_wide_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, float* lse, const WideParams& p, int grid,
                            cudaStream_t stream, const DeviceInfo& dev) {
    using C = WideCfg<D>;
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_fwd_wide_kernel<D, OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    attn_fwd_wide_kernel<D, OUT_F32, VARLEN><<<(unsigned)grid, kWThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, to, lse, p, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

uint32_t next_wide_queue_slot() {
    static std::atomic<uint32_t> launches{0};
    return launches.fetch_add(1u, std::memory_order_relaxed) % kWideQueueSlots;
}

}  // namespace

attn_status_t launch_fwd_wide(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                              attn_out_dtype_t o_dtype, cudaStream_t stream, const DeviceInfo& dev) {
    WideParams p;
    // units are single 128-row Q tiles
    p.shape = make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal, dev.num_sms, kWM);
    if (p.shape.units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    p.group = Hq / Hkv;
    p.off = Nk - Nq;
    p.d_act = d;
    p.c = scale * kWLog2e;
    p.o = o;
    p.cu_q = nullptr;
    p.cu_k = nullptr;
    p.total_q = 0;
    p.total_k = 0;
    p.slot = next_wide_queue_slot();
    const long long units = p.shape.units;
    const int grid = (int)(units < dev.num_sms ? units : dev.num_sms);
    CUtensorMap tq, tk, tv, to;
    attn_status_t st;
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if ((st = encode_tmap_bf16_3d(&tq, q, d, Nq, (long long)B * Hq, kWM)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tk, k, d, Nk, (long long)B * Hkv, kWN)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tv, v, d, Nk, (long long)B * Hkv, kWV)) != ATTN_OK) return st;
    if ((st = encode_tmap_out_3d(&to, o, f32, d, Nq, (long long)B * Hq, wide_epi_cols(f32), 32)) != ATTN_OK)
        return st;
    if (d <= 192)
        return f32 ? launch_wide_t<192, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
                   : launch_wide_t<192, false>(tq, tk, tv, to, lse, p, grid, stream, dev);
    return f32 ? launch_wide_t<256, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
               : launch_wide_t<256, false>(tq, tk, tv, to, lse, p, grid, stream, dev);
}

attn_status_t launch_fwd_wide_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const int* cu_q, const int* cu_k, int B, int Hq, int Hkv,
                                     int total_q, int total_k, int max_q, int max_k, int d,
                                     int causal, float scale, attn_out_dtype_t o_dtype,
                                     cudaStream_t stream, const DeviceInfo& dev) {
    WideParams p;
    // units cover every sequence at the maximum lengths; the producer skips
    // the Q tiles past each sequence's own length
    p.shape = make_fwd_shape(B, Hq, Hkv, max_q, max_k, d, causal, 0, kWM);
    if (p.shape.units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    p.group = Hq / Hkv;
    p.off = 0;
    p.d_act = d;
    p.c = scale * kWLog2e;
    p.o = o;
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.slot = next_wide_queue_slot();
    const long long units = p.shape.units;
    const int grid = (int)(units < dev.num_sms ? units : dev.num_sms);
    CUtensorMap tq, tk, tv, to;
    attn_status_t st;
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if ((st = encode_tmap_ragged(&tq, q, false, d, Hq, 64, kWM, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tk, k, false, d, Hkv, 64, kWN, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tv, v, false, d, Hkv, 64, kWV, true)) != ATTN_OK) return st;
    // (O is written from registers, never by this map; it is still encoded,
    // which checks O's alignment like the other maps)
    if ((st = encode_tmap_ragged(&to, o, f32, d, Hq, wide_epi_cols(f32), 32, false)) != ATTN_OK) return st;
    if (d <= 192)
        return f32 ? launch_wide_t<192, true, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
                   : launch_wide_t<192, false, true>(tq, tk, tv, to, lse, p, grid, stream, dev);
    return f32 ? launch_wide_t<256, true, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
               : launch_wide_t<256, false, true>(tq, tk, tv, to, lse, p, grid, stream, dev);
}

}  // namespace gb300
