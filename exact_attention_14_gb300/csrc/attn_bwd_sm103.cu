// attn_bwd_sm103.cu -- attention backward (dQ, dK, dV) for sm_103a.
//
// Method: lecture notes "Optimizing Attention for Modern Hardware:
// FlashAttention 1-4", 2.6 (P recomputed from the stored logsumexp,
// D = rowsum(dO o O), the K/V-outer loop with dK and dV accumulated on chip and
// dQ accumulated with atomic adds) and exercise 6; "Flash Attention 3/4
// notes", FA4 section 2 (five MMAs per tile -- S, dP, dV, dK, dQ -- with the
// accumulators in tensor memory).
//
// Three kernels, none of them with atomics (exercise 6 weighs K/V-outer with
// dQ atomics against Q-outer with dK/dV atomics; this build runs one pass of
// each loop order instead, recomputing S and dP in both: seven products per
// tile pair instead of five, and every gradient written once, bit-identical
// from run to run):
//  prep  per query row: D = sum_c dO_c O_c and lse2 = LSE log2(e), padded to
//        whole 128-row tiles (lse2 = +inf and D = 0 past Nq, so padded rows
//        get P = 0 and dS = 0).
//  dkdv  one item per (b, KV head g, 128-key tile).  K and V of the tile stay
//        in shared memory; the item walks every query head of g's group and
//        every 128-row Q tile that can see its keys.  Per Q tile:
//          S^T  = K Q^T,  dP^T = V dO^T      (tcgen05, operands K-major in smem)
//          P^T  = 2^(S^T c - lse2),  dS^T = P^T o (dP^T - D)
//                 (warps 4-11, one key row per thread and half of the
//                 tile's query columns per warpgroup; P^T and dS^T go to
//                 TMEM as bf16 pairs)
//          dV  += P^T dO,  dK += dS^T Q      (A from TMEM, B MN-major in smem)
//        After the last tile dK (times scale) and dV are written once (at
//        d = 128 through tensor stores from each warp's 4 KiB of staging).
//  dq    one item per (b, query head, 128-row Q tile), K/V tiles streamed
//        through a ring.  Per K/V tile:
//          S = Q K^T,  dP = dO V^T,  dS = P o (dP - D)  (one query row per
//          thread and half of the tile's keys per warpgroup, its lse2 and D
//          in registers; dS to TMEM over S)
//          dQ += dS K                        (A from TMEM, B = K MN-major)
//        After the last tile dQ (times scale) is written once.
//
// Both passes run persistent grids of at most one CTA per SM; CTA c takes items
// c, c + gridDim.x, ... and its roles run from one item into the next: the
// producer loads the next item's K and V (dkdv) or Q and dO (dq) as soon as
// the current item's last products that read them complete, the rings and
// the TMEM buffers keep counting across items, and an item's first
// accumulating product waits only for its first P^T / dS, which the
// elementwise warps form after reading out the previous item's accumulators.
//
// Roles (12 warps): warp 0 TMA producer, warp 1 MMA issuer and TMEM owner,
// warps 2-3 idle, warps 4-7 and 8-11 the elementwise work, two warpgroups
// (one TMEM lane quarter per warp; warpgroup h takes f32 columns
// [64h, 64h + 64) of S^T / dP^T / S / dP and writes their bf16 pairs to
// columns [64h, 64h + 32), over columns it has read itself).  The d > 128
// passes further down keep 8 warps, one elementwise warpgroup.
//
// TMEM, dkdv (512 columns): [0,128) S^T, then P^T in [0,32) and [64,96);
// [128,256) dP^T, then dS^T in [128,160) and [192,224); dV [256,256+d); dK
// [256+d,256+2d).  The P^T / dS^T
// warps work in two phases per Q tile (P^T from S^T, then dS^T from dP^T), and
// the MMAs interleave with them: dV(i) and S^T(i+1) run during phase 2 of tile
// i, dK(i) and dP^T(i+1) during phase 1 of tile i+1 (each next-tile product is
// issued after the one that reads its columns: one CTA's MMAs run in issue
// order).
// TMEM, dq: S in [0,128) for even K/V tiles and [384,512) for odd ones (dS over
// its columns [0,32) and [64,96)), dP [128,256), dQ [256,256+d).  K streams through a
// 3-stage ring and V through a 2-stage one; S_{j+2} is issued as soon as dQ_j
// has read tile j's S buffer, so the dS warps' exponentials for tile j+1
// (phase 1) overlap dQ_j and dP_{j+1}.
#include <cmath>
#include <cstdint>

#include "fwd_sched.h"
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kBwdThreads = 256;    // the d > 128 passes: producer, MMA, one P/dS warpgroup
constexpr int kBwdThreadsEw = 384;  // the d <= 128 passes: producer, MMA, two P/dS warpgroups
constexpr int kBT = 128;  // keys per K/V tile, query rows per Q tile
constexpr float kBwdLog2e = 1.44269504088896340736f;
constexpr int kMaxSmemPerBlock = 232448;

template <int D>
struct BwdCfg {
    static constexpr int kTile = kBT * D * 2;   // one 128-row bf16 tile
    static constexpr int kK = 0;
    static constexpr int kV = kTile;
    static constexpr int kQ = 2 * kTile;        // 2 stages
    static constexpr int kDO = 4 * kTile;       // 2 stages
    static constexpr int kStg = 6 * kTile;      // 8 P/dS warps x 4 KiB: dK / dV store staging
    static constexpr int kLD = kStg + 8 * 4096; // 2 stages x (lse2[128], D[128])
    static constexpr int kBar = kLD + 2 * 1024;
    static constexpr int kLayout = kBar + 256;
    static constexpr int kSmemBytes =
        kLayout + 1024 < kMaxSmemPerBlock ? kLayout + 1024 : kMaxSmemPerBlock;
    static_assert(kLayout <= kMaxSmemPerBlock, "shared memory budget");
};

struct BwdParams {
    int B, Hq, Hkv, Nq, Nk, Nq_pad, group, off, n_kt, causal;
    int sec_groups;     // (b, KV head) groups per L2 section
    int d_act;          // the tensors' head dim (<= D; the tiles' columns past it are zeros)
    float c;      // scale * log2(e)
    float scale;
    const float* lse2;  // [B*Hq, Nq_pad]; packed batches [Hq, vstride]
    const float* dvec;  // [B*Hq, Nq_pad]; packed batches [Hq, vstride]
    void* dq;           // [B, Hq, Nq, d]; packed batches [total_q, Hq, d]
    void* dk;           // [B, Hkv, Nk, d]; packed batches [total_k, Hkv, d]
    void* dv;
    // packed batches (the VARLEN instantiations): Nq and Nk above are the
    // longest lengths; sequence b holds rows [cu_q[b], cu_q[b+1]) of q / o / dO
    // / dQ and [cu_k[b], cu_k[b+1]) of k / v / dK / dV; its rows of lse2 / dvec
    // start at varlen_vbase(cu_q[b], b) of each head's vstride rows.
    const int* cu_q;
    const int* cu_k;
    int total_q, total_k, vstride;
};

// Row of sequence b's first query in a head's rows of lse2 / dvec for packed
// batches: the packed row rounded up to 4 floats (16-byte bulk copies), plus
// 132 rows per earlier sequence, so that each sequence's rows padded to whole
// 128-row tiles never reach the next sequence's.
__host__ __device__ inline int varlen_vbase(int q_row0, int b) { return ((q_row0 + 3) & ~3) + 132 * b; }

// Sequence b of a packed batch: first rows and lengths.  False when its
// offsets leave the arrays, decrease, exceed the longest length, give query
// rows without keys, or (causal) more queries than keys: the checks of the
// packed forward.
__device__ __forceinline__ bool bwd_varlen_seq(const BwdParams& p, int b, int& q0, int& nq,
                                               int& k0, int& nk) {
    const int qs = __ldg(p.cu_q + b), qe = __ldg(p.cu_q + b + 1);
    const int ks = __ldg(p.cu_k + b), ke = __ldg(p.cu_k + b + 1);
    q0 = qs; nq = qe - qs; k0 = ks; nk = ke - ks;
    return 0 <= qs && qs <= qe && qe <= p.total_q && qe - qs <= p.Nq && 0 <= ks && ks <= ke &&
           ke <= p.total_k && ke - ks <= p.Nk && (qe == qs || ke > ks) &&
           (!p.causal || qe - qs <= ke - ks);
}

struct __align__(8) BwdBars {
    uint64_t kv_full, kv_empty;  // K and V of an item; read by its last S^T and dP^T
    uint64_t qd_full[2], qd_empty[2];
    uint64_t s_full, dp_full, p_full, ds_full, acc_full, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

// The CTA's work: K/V tile kt of (b, g) and the Q tiles [qt_first, n_qt) of
// each query head of the group, head-major.
//
// Order of the CTAs: the (b, KV head) groups are cut into L2 sections whose
// Q, dO, K and V fit an L2 budget (so each Q / dO tile is read from DRAM once
// for all the section's key tiles); sections run in order, and inside a
// section key tiles are outer (causal tile 0, which sees the most query
// tiles, first).
struct BwdWork {
    int b, g, kt, k0, qt_first, n_qt_cta, n_tiles;
    // the (b, g) problem: lengths, causal offset, and for packed batches the
    // sequence's first rows (in q and k) and its rows of lse2 / dvec
    int nq, nk, off, qb, kb, vbase;
};

__device__ __forceinline__ BwdWork bwd_work(const BwdParams& p, unsigned idx) {
    BwdWork w;
    const unsigned all = (unsigned)(p.B * p.Hkv);
    const unsigned S = (unsigned)p.sec_groups;
    const unsigned per_sec = S * (unsigned)p.n_kt;
    const unsigned sec = idx / per_sec;
    const unsigned r = idx - sec * per_sec;
    const unsigned rest = all - sec * S;
    const unsigned gs = rest < S ? rest : S;  // groups in this (possibly partial) section
    w.kt = (int)(r / gs);
    const int bg = (int)(sec * S + (r - (unsigned)w.kt * gs));
    w.b = bg / p.Hkv;
    w.g = bg - w.b * p.Hkv;
    w.k0 = w.kt * kBT;
    const int n_qt = (p.Nq + kBT - 1) / kBT;
    int first = 0;
    if (p.causal) {
        const int lo = w.k0 - p.off;  // the first query that sees key k0
        first = lo <= 0 ? 0 : lo / kBT;
    }
    w.qt_first = first;
    w.n_qt_cta = n_qt - first > 0 ? n_qt - first : 0;
    w.n_tiles = w.n_qt_cta * p.group;
    w.nq = p.Nq;
    w.nk = p.Nk;
    w.off = p.off;
    w.qb = w.kb = w.vbase = 0;
    return w;
}

// The same for packed batches: item index = (b * Hkv + g) * n_kt + kt, n_kt
// for the longest key length.  Key tiles past a sequence's end, and every tile
// of a sequence whose offsets fail the checks (reported in the error word),
// have no work and write nothing.
__device__ __forceinline__ BwdWork bwd_work_varlen(const BwdParams& p, unsigned idx, unsigned int* err) {
    BwdWork w;
    const int per_b = p.Hkv * p.n_kt;
    w.b = (int)idx / per_b;
    const int rem = (int)idx - w.b * per_b;
    w.g = rem / p.n_kt;
    w.kt = rem - w.g * p.n_kt;
    w.k0 = w.kt * kBT;
    int q0, nq, k0, nk;
    if (!bwd_varlen_seq(p, w.b, q0, nq, k0, nk)) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadSeqlen);
        q0 = nq = k0 = nk = 0;
    }
    w.nq = nq;
    w.nk = nk;
    w.off = nk - nq;
    w.qb = q0;
    w.kb = k0;
    w.vbase = varlen_vbase(q0, w.b);
    const int n_qt = (nq + kBT - 1) / kBT;
    int first = 0;
    if (p.causal) {
        const int lo = w.k0 - w.off;
        first = lo <= 0 ? 0 : lo / kBT;
    }
    w.qt_first = first;
    w.n_qt_cta = (w.k0 < nk && n_qt - first > 0) ? n_qt - first : 0;
    w.n_tiles = w.n_qt_cta * p.group;
    return w;
}

// The dK/dV pass runs a persistent grid (at most one CTA per SM): CTA c takes
// items c, c + gridDim.x, ... of the order above, each one key tile, and
// keeps its pipeline running from one item into the next.
template <bool VARLEN>
__device__ __forceinline__ BwdWork bwd_item(const BwdParams& p, unsigned idx, unsigned int* err) {
    if constexpr (VARLEN) return bwd_work_varlen(p, idx, err);
    else return bwd_work(p, idx);
}

__device__ __forceinline__ void bwd_abort(BwdBars* bars, unsigned int* err) {
    atomicOr(err, kErrTimeout);
    *((volatile int*)&bars->abort) = 1;
}

// ---------------------------------------------------------------------------
// Producer
// ---------------------------------------------------------------------------
template <int D, bool VARLEN>
__device__ void bwd_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                             const CUtensorMap* tdo, uint8_t* smem, BwdBars* bars,
                             const BwdParams& p, unsigned n_items, unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    bool ok = true;
    int issued = 0;   // Q / dO tiles issued, over the CTA's items
    int kv_uses = 0;  // K / V loads issued (items with work)
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const BwdWork w = bwd_item<VARLEN>(p, idx, err);
        if (w.n_tiles == 0) continue;
        // K and V of the item, once the previous item's last S^T and dP^T have
        // read theirs
        if (kv_uses > 0)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->kv_empty), (kv_uses - 1) & 1, abort_flag));
        if (!ok) break;
        // K/V head: an index into [B * Hkv], or into [Hkv] of the packed rows
        const int kvh = VARLEN ? w.g : w.b * p.Hkv + w.g;
        if (leader) {
            const uint32_t bar = smem_u32(&bars->kv_full);
            mbar_arrive_expect_tx(bar, 2 * C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                if constexpr (VARLEN) {
                    const int r = kRaggedWindow - w.nk + w.k0;
                    tma_load_5d(smem_u32(smem + C::kK) + c * 16384, tk, bar, 64 * c, kvh, r, w.kb + w.nk,
                                kRaggedWindow);
                    tma_load_5d(smem_u32(smem + C::kV) + c * 16384, tv, bar, 64 * c, kvh, r, w.kb + w.nk,
                                kRaggedWindow);
                } else {
                    tma_load_3d(smem_u32(smem + C::kK) + c * 16384, tk, bar, 64 * c, w.k0, kvh);
                    tma_load_3d(smem_u32(smem + C::kV) + c * 16384, tv, bar, 64 * c, w.k0, kvh);
                }
            }
        }
        __syncwarp();
        ++kv_uses;
        for (int i = 0; i < w.n_tiles && ok; ++i) {
            const int st = issued & 1;
            if (issued >= 2)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->qd_empty[st]), ((issued >> 1) - 1) & 1,
                                                       abort_flag));
            if (!ok) break;
            const int hq = w.g * p.group + i / w.n_qt_cta;
            const int q0 = (w.qt_first + i % w.n_qt_cta) * kBT;
            const int bh = w.b * p.Hq + hq;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->qd_full[st]);
                mbar_arrive_expect_tx(bar, 2 * C::kTile + 1024);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if constexpr (VARLEN) {
                        const int r = kRaggedWindow - w.nq + q0;
                        tma_load_5d(smem_u32(smem + C::kQ + st * C::kTile) + c * 16384, tq, bar, 64 * c, hq, r,
                                    w.qb + w.nq, kRaggedWindow);
                        tma_load_5d(smem_u32(smem + C::kDO + st * C::kTile) + c * 16384, tdo, bar, 64 * c, hq,
                                    r, w.qb + w.nq, kRaggedWindow);
                    } else {
                        tma_load_3d(smem_u32(smem + C::kQ + st * C::kTile) + c * 16384, tq, bar, 64 * c, q0,
                                    bh);
                        tma_load_3d(smem_u32(smem + C::kDO + st * C::kTile) + c * 16384, tdo, bar, 64 * c, q0,
                                    bh);
                    }
                }
                const size_t row = VARLEN ? (size_t)hq * p.vstride + (size_t)(w.vbase + q0)
                                          : (size_t)bh * p.Nq_pad + q0;
                bulk_load(smem_u32(smem + C::kLD + st * 1024), p.lse2 + row, 512, bar);
                bulk_load(smem_u32(smem + C::kLD + st * 1024 + 512), p.dvec + row, 512, bar);
            }
            __syncwarp();
            ++issued;
        }
    }
    if (!ok && leader) bwd_abort(bars, err);
    // Drain: every issued copy lands before the CTA may exit.
    if (kv_uses > 0) mbar_wait(smem_u32(&bars->kv_full), (kv_uses - 1) & 1, nullptr);
    for (int st = 0; st < 2 && st < issued; ++st) {
        const int uses = (issued - st + 1) / 2;
        mbar_wait(smem_u32(&bars->qd_full[st]), (uses - 1) & 1, nullptr);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer
// ---------------------------------------------------------------------------
constexpr uint32_t kBwdDescHi = sdesc_hi_sw128(1024);

// M=128 x N=128 x K=d, both operands K-major (SW128, 64-column chunks 16 KiB
// apart): S^T = K Q^T or dP^T = V dO^T.
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t step = (kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4);
        mma_ss_warp(d_tmem, sdesc_join(a_lo + step, kBwdDescHi), sdesc_join(b_lo + step, kBwdDescHi),
                    idesc, kk > 0 ? 1u : 0u);
    }
}

// M=128 x N=d x K=128 with A from TMEM and B MN-major in smem (16 rows of
// 128 B per K=16): dV += P^T dO, dK += dS^T Q or dQ += dS K.  A is bf16 pairs,
// 8 columns per K=16, in two blocks of 32 columns: K [0, 64) at a_tmem and
// [64, 128) at a_tmem + 64, each written by the warpgroup that owns those
// f32 columns (a_chunk_col), over columns it has read.
__device__ __forceinline__ uint32_t a_chunk_col(int cc) { return (uint32_t)((cc >> 1) * 64 + (cc & 1) * 16); }

__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kBT / 16; ++kk)
        mma_ts_warp(d_tmem, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8,
                    sdesc_join(b_lo + kk * (2048 >> 4), kBwdDescHi), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, bool VARLEN>
__device__ void bwd_mma(uint8_t* smem, BwdBars* bars, uint32_t tmem, const BwdParams& p,
                        unsigned n_items, unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idS = make_idesc_bf16(128, 128, 0, 0);
    const uint32_t idKV = make_idesc_bf16(128, D, 0, 1);
    const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
    const uint32_t k_kmaj = sdesc_lo(smem_u32(smem + C::kK), 16);
    const uint32_t v_kmaj = sdesc_lo(smem_u32(smem + C::kV), 16);
    auto q_kmaj = [&](int st) { return sdesc_lo(smem_u32(smem + C::kQ + st * C::kTile), 16); };
    auto do_kmaj = [&](int st) { return sdesc_lo(smem_u32(smem + C::kDO + st * C::kTile), 16); };
    auto q_mn = [&](int st) { return sdesc_lo(smem_u32(smem + C::kQ + st * C::kTile), 16384); };
    auto do_mn = [&](int st) { return sdesc_lo(smem_u32(smem + C::kDO + st * C::kTile), 16384); };
    auto wait_all = [&](uint32_t bar, uint32_t parity, int polls) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, polls));
    };
    bool ok = true;
    int g = 0;  // Q / dO tiles consumed, over the CTA's items
    int u = 0;  // items with work
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const BwdWork w = bwd_item<VARLEN>(p, idx, err);
        const int n = w.n_tiles;
        if (n == 0) continue;
        ok = wait_all(smem_u32(&bars->kv_full), u & 1, 0) &&
             wait_all(smem_u32(&bars->qd_full[g & 1]), (g >> 1) & 1, 0);
        if (!ok) break;
        // S^T and dP^T of the item's first tile: their columns were last read
        // by the previous item's dV and dK, issued before (one CTA's MMAs run
        // in issue order); its dV and dK (accumulate = 0) wait for P^T and
        // dS^T, which the P/dS warps write after reading out the previous
        // item's dV and dK.
        tc_fence_after();
        issue_kmajor<D>(tS, k_kmaj, q_kmaj(g & 1), idS);
        mma_commit_warp(smem_u32(&bars->s_full));
        issue_kmajor<D>(tdP, v_kmaj, do_kmaj(g & 1), idS);
        mma_commit_warp(smem_u32(&bars->dp_full));
        if (n == 1) mma_commit_warp(smem_u32(&bars->kv_empty));  // K and V are read
        // Per Q tile i: dV(i) once P^T(i) is in TMEM, then S^T(i+1) into the
        // columns dV(i) has read; dK(i) once dS^T(i) is in TMEM, then dP^T(i+1)
        // into the columns dK(i) has read.  The P^T / dS^T warps work on tile i
        // while the tensor cores run dV(i), S^T(i+1) and then dK(i), dP^T(i+1).
        for (int i = 0; i < n && ok; ++i) {
            const int gi = g + i;
            const int st = gi & 1;
            const int st1 = (gi + 1) & 1;
            const bool more = i + 1 < n;
            ok = wait_all(smem_u32(&bars->p_full), gi & 1, 32);
            if (!ok) break;
            tc_fence_after();
            issue_tmem_a(tdV, tS, do_mn(st), idKV, i > 0);          // dV += P^T dO
            if (more) {
                ok = wait_all(smem_u32(&bars->qd_full[st1]), ((gi + 1) >> 1) & 1, 0);
                if (!ok) break;
                tc_fence_after();
                issue_kmajor<D>(tS, k_kmaj, q_kmaj(st1), idS);       // S^T(i+1)
                mma_commit_warp(smem_u32(&bars->s_full));
            }
            ok = wait_all(smem_u32(&bars->ds_full), gi & 1, 32);
            if (!ok) break;
            tc_fence_after();
            issue_tmem_a(tdK, tdP, q_mn(st), idKV, i > 0);          // dK += dS^T Q
            mma_commit_warp(smem_u32(&bars->qd_empty[st]));         // Q and dO of tile i are read
            if (more) {
                issue_kmajor<D>(tdP, v_kmaj, do_kmaj(st1), idS);     // dP^T(i+1)
                mma_commit_warp(smem_u32(&bars->dp_full));
                if (i + 2 == n) mma_commit_warp(smem_u32(&bars->kv_empty));  // the last S^T, dP^T
            }
        }
        if (ok) mma_commit_warp(smem_u32(&bars->acc_full));
        g += n;
        ++u;
    }
    if (!ok && leader) bwd_abort(bars, err);
    // Drain: all issued MMAs complete before TMEM is released.
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// ---------------------------------------------------------------------------
// P / dS warpgroups (one key row per thread, half the columns each) and the
// dK / dV epilogue
// ---------------------------------------------------------------------------
// P^T = 2^(S^T c - lse2) for 32 query columns [qc, qc + 32) of this thread's
// key row, kept in fp32 (pf) and packed to bf16 pairs (pp).  lim: query column
// qc + x is allowed iff qc + x >= lim (causal), else all.  The tile's lse2
// comes from shared memory 4 at a time (broadcast).
template <bool MASKED>
__device__ __forceinline__ void p_chunk(const uint32_t (&s)[32], uint32_t lse2s, int qc, float c,
                                        int lim, float (&pf)[32], uint32_t (&pp)[16]) {
    const uint64_t c2 = f2(c, c);
#pragma unroll
    for (int x4 = 0; x4 < 8; ++x4) {
        const float4 l4 = lds128_f32(lse2s + 4u * (qc + 4 * x4));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int x = 2 * x4 + h;
            const int q = qc + 2 * x;
            const uint64_t nl = h == 0 ? f2(-l4.x, -l4.y) : f2(-l4.z, -l4.w);
            float a0, a1;
            f2_split(f2_fma(f2(__uint_as_float(s[2 * x]), __uint_as_float(s[2 * x + 1])), c2, nl), a0, a1);
            float p0 = ex2(a0), p1 = ex2(a1);
            if constexpr (MASKED) {
                p0 = q >= lim ? p0 : 0.f;
                p1 = q + 1 >= lim ? p1 : 0.f;
            }
            pf[2 * x] = p0;
            pf[2 * x + 1] = p1;
            pp[x] = pack_bf16x2(p0, p1);
        }
    }
}

// dS^T = P^T o (dP^T - D) for the same 32 query columns, packed to bf16 pairs.
__device__ __forceinline__ void ds_chunk_t(const float (&pf)[32], const uint32_t (&dp)[32],
                                           uint32_t ds_vec, int qc, uint32_t (&dd)[16]) {
#pragma unroll
    for (int x4 = 0; x4 < 8; ++x4) {
        const float4 d4 = lds128_f32(ds_vec + 4u * (qc + 4 * x4));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int x = 2 * x4 + h;
            const uint64_t nd = h == 0 ? f2(-d4.x, -d4.y) : f2(-d4.z, -d4.w);
            float d0, d1;
            f2_split(f2_mul(f2(pf[2 * x], pf[2 * x + 1]),
                            f2_add(f2(__uint_as_float(dp[2 * x]), __uint_as_float(dp[2 * x + 1])), nd)),
                     d0, d1);
            dd[x] = pack_bf16x2(d0, d1);
        }
    }
}

// Store of 32 columns [cc, cc + 32) of this warp's 32 rows of an output
// (rows row0 .. row0 + 31 of a row-major array with `row_elems` elements per
// row), whole 32-byte sectors per store: lanes 2k and 2k+1 swap one 16-byte
// piece of each sector, then both write row 2k's sector and, in the next
// store, row 2k+1's.  Run by the whole warp (shuffles); rows at or past
// rows_live and columns at or past ncols (uniform, a multiple of 8) are not
// written.
template <bool OUT_F32>
__device__ __forceinline__ void store_rows32_pairs(void* base, size_t row0, size_t row_elems, int cc,
                                                   const float (&v)[32], int ncols, int rows_live,
                                                   int lane) {
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
    uint8_t* b8 = static_cast<uint8_t*>(base);
    uint8_t* pa = b8 + ((row0 + (size_t)ra) * row_elems + (size_t)cc) * kEs + (odd ? 16 : 0);
    uint8_t* pb = b8 + ((row0 + (size_t)rb) * row_elems + (size_t)cc) * kEs + (odd ? 16 : 0);
    const bool live_a = ra < rows_live, live_b = rb < rows_live;
#pragma unroll
    for (int sct = 0; sct < kPieces / 2; ++sct) {
        if (2 * sct * kColsPerPiece >= ncols) break;
        const int pe = 2 * sct, po = 2 * sct + 1;
        const bool col_ok = (odd ? po : pe) * kColsPerPiece < ncols;
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
__device__ void bwd_pds(int wq, int grp, int lane, uint8_t* smem, BwdBars* bars, uint32_t tmem,
                        const CUtensorMap* tdk, const CUtensorMap* tdv, const BwdParams& p,
                        unsigned n_items, unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + 128 + lane_off;
    const int j = wq * 32 + lane;  // key row of the tile
    // this warpgroup's half of the output columns
    const int cc_lo = grp * (D / 2), cc_hi = cc_lo + D / 2;
    bool ok = true;
    int g = 0;  // Q tiles done, over the CTA's items
    int u = 0;  // items with work
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const BwdWork w = bwd_item<VARLEN>(p, idx, err);
        const int jg = w.k0 + j;
        for (int i = 0; i < w.n_tiles && ok; ++i) {
            const int gi = g + i;
            const int st = gi & 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->s_full), gi & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            const int q0 = (w.qt_first + i % w.n_qt_cta) * kBT;
            const uint32_t lse2s = smem_u32(smem + C::kLD + st * 1024);
            const uint32_t ds_vec = lse2s + kBT * 4;
            // causal: query q0 + x sees key jg iff x >= jg - off - q0
            const int lim = jg - w.off - q0;
            const bool masked = p.causal && (q0 + w.off < w.k0 + kBT - 1);
            // Phase 1: P^T from S^T for this warpgroup's 64 query columns, kept
            // in registers and written as bf16 over the S^T columns it has read;
            // with the other warpgroup's, releases dV(i) and S^T(i+1).
            float pf0[32], pf1[32];
            auto phase1 = [&](int cc, float (&pf)[32]) {
                uint32_t sv[32], pp[16];
                tmem_ld32(tS + cc * 32, sv);
                tmem_wait_ld();
                if (masked)
                    p_chunk<true>(sv, lse2s, cc * 32, p.c, lim, pf, pp);
                else
                    p_chunk<false>(sv, lse2s, cc * 32, p.c, lim, pf, pp);
                tmem_st16(tS + a_chunk_col(cc), pp);
            };
            phase1(2 * grp, pf0);
            phase1(2 * grp + 1, pf1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
            // Phase 2: dS^T from P^T and dP^T, written as bf16 over the dP^T
            // columns already read; releases dK(i) and dP^T(i+1).
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->dp_full), gi & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            auto phase2 = [&](int cc, const float (&pf)[32]) {
                uint32_t dp[32], dd[16];
                tmem_ld32(tdP + cc * 32, dp);
                tmem_wait_ld();
                ds_chunk_t(pf, dp, ds_vec, cc * 32, dd);
                tmem_st16(tdP + a_chunk_col(cc), dd);
            };
            phase2(2 * grp, pf0);
            phase2(2 * grp + 1, pf1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&bars->ds_full));
                mbar_arrive(smem_u32(&bars->qd_empty[st]));
            }
        }
        if (!ok) break;
        // dK = scale * dS^T Q, dV = P^T dO: one key row per thread, written once
        // this warp's first key row and how many of its rows are inside Nk
        // (packed batches: rows of Hkv * d elements, the head's d columns at
        // offset g * d)
        const size_t wrow0 = VARLEN ? (size_t)(w.kb + w.k0 + wq * 32)
                                    : ((size_t)w.b * p.Hkv + w.g) * p.Nk + (size_t)(w.k0 + wq * 32);
        const int rows_live = w.nk - (w.k0 + wq * 32);
        const size_t row_elems = VARLEN ? (size_t)p.Hkv * p.d_act : (size_t)p.d_act;
        const size_t head_off = VARLEN ? (size_t)w.g * p.d_act * (OUT_F32 ? 4 : 2) : 0;
        void* dk_base = static_cast<uint8_t*>(p.dk) + head_off;
        void* dv_base = static_cast<uint8_t*>(p.dv) + head_off;
        if (w.n_tiles == 0) {
            float z[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) z[x] = 0.f;
#pragma unroll 1
            for (int cc = cc_lo; cc < cc_hi && cc < p.d_act; cc += 32) {
                const int nc = p.d_act - cc < 32 ? p.d_act - cc : 32;
                store_rows32_pairs<OUT_F32>(dk_base, wrow0, row_elems, cc, z, nc, rows_live, lane);
                store_rows32_pairs<OUT_F32>(dv_base, wrow0, row_elems, cc, z, nc, rows_live, lane);
            }
            continue;
        }
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->acc_full), u & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        // The next item's dV and dK (accumulate = 0) are issued only after this
        // warpgroup's next P^T arrival, which follows these reads.
        if constexpr (D == 128) {
            // dV, then dK (x scale): boxes of 32 rows x 128 bytes written into the
            // warp's 4 KiB of shared memory (128-byte swizzle) and stored by the
            // tensor-memory accelerator, so the stores drain while the next item
            // runs; a box waits only until the warp's previous one has been read.
            constexpr int kBoxCols = OUT_F32 ? 32 : 64;
            const uint32_t stg = smem_u32(smem + C::kStg + (grp * 4 + wq) * 4096);
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const float sc = t ? p.scale : 1.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D / 2; c0 += kBoxCols) {
                    uint32_t wv[32];
#pragma unroll
                    for (int c = 0; c < kBoxCols; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(tmem + 256 + t * D + cc_lo + c0 + c + lane_off, r);
                        tmem_wait_ld();
                        if constexpr (OUT_F32) {
#pragma unroll
                            for (int x = 0; x < 32; ++x) wv[x] = __float_as_uint(__uint_as_float(r[x]) * sc);
                        } else {
#pragma unroll
                            for (int x = 0; x < 16; ++x)
                                wv[c / 2 + x] = pack_bf16x2(__uint_as_float(r[2 * x]) * sc,
                                                            __uint_as_float(r[2 * x + 1]) * sc);
                        }
                    }
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sts128(stg + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4)), wv[4 * j], wv[4 * j + 1],
                               wv[4 * j + 2], wv[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const CUtensorMap* map = t ? tdk : tdv;
                        const int col = cc_lo + c0;
                        if constexpr (VARLEN)
                            tma_store_5d(map, stg, col, w.g, kRaggedWindow - w.nk + w.k0 + wq * 32, w.kb + w.nk,
                                         kRaggedWindow);
                        else
                            tma_store_3d(map, stg, col, w.k0 + wq * 32, w.b * p.Hkv + w.g);
                        bulk_commit_group();
                    }
                }
            }
        } else {
#pragma unroll 1
        for (int cc = cc_lo; cc < cc_hi; cc += 32) {
            uint32_t r[32];
            float v[32];
            tmem_ld32(tmem + 256 + cc + lane_off, r);
            tmem_wait_ld();
            const int nc = p.d_act - cc < 32 ? p.d_act - cc : 32;  // <= 0: past the head dim
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]);
            if (nc > 0) store_rows32_pairs<OUT_F32>(dv_base, wrow0, row_elems, cc, v, nc, rows_live, lane);
            tmem_ld32(tmem + 256 + D + cc + lane_off, r);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]) * p.scale;
            if (nc > 0) store_rows32_pairs<OUT_F32>(dk_base, wrow0, row_elems, cc, v, nc, rows_live, lane);
        }
        }
        tc_fence_before();
        g += w.n_tiles;
        ++u;
    }
    if (!ok) bwd_abort(bars, err);
    // every staged store has read shared memory and written global memory
    // before the CTA may exit
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
}

template <int D, bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreadsEw, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                     const BwdParams p, unsigned int* err) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
    // The layout must fit the allocation after the alignment (checked, not assumed).
    if ((uintptr_t)(smem - smem_raw) + C::kLayout > (uintptr_t)C::kSmemBytes) {
        if (threadIdx.x == 0) atomicOr(err, kErrLayout);
        return;
    }
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::kBar);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned n_items = (unsigned)(p.B * p.Hkv * p.n_kt);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        mbar_init(smem_u32(&bars->kv_empty), 1);  // the commit after an item's last S^T and dP^T
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->qd_full[s]), 1);
            mbar_init(smem_u32(&bars->qd_empty[s]), 1 + 8);  // dK commit + 8 P/dS warps
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->p_full), 8);
        mbar_init(smem_u32(&bars->ds_full), 8);
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) bwd_producer<D, VARLEN>(&tq, &tk, &tv, &tdo, smem, bars, p, n_items, err);
    else if (warp == 1) bwd_mma<D, VARLEN>(smem, bars, tmem, p, n_items, err);
    else if (warp >= 4)
        bwd_pds<D, OUT_F32, VARLEN>(warp & 3, (warp - 4) >> 2, lane, smem, bars, tmem, &tdk, &tdv, p, n_items, err);

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// dQ pass (Q-outer)
// ---------------------------------------------------------------------------
template <int D>
struct DqCfg {
    static constexpr int kTile = kBT * D * 2;
    static constexpr int kQ = 0;
    static constexpr int kDO = kTile;
    static constexpr int kKRing = 2 * kTile;    // 3 stages of K
    static constexpr int kVRing = 5 * kTile;    // 2 stages of V
    static constexpr int kBar = 7 * kTile;
    static constexpr int kLayout = kBar + 256;
    static constexpr int kSmemBytes =
        kLayout + 1024 < kMaxSmemPerBlock ? kLayout + 1024 : kMaxSmemPerBlock;
    static_assert(kLayout <= kMaxSmemPerBlock, "shared memory budget");
};

struct __align__(8) DqBars {
    uint64_t q_full, q_empty;  // Q and dO of an item; read by its last S and dP
    uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
    uint64_t s_full[2], dp_full, ds_full, dq_full, drain;  // s_full[b]: the S in buffer b
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(DqBars) <= 256, "barrier block");

// The CTA's Q tile and the K/V tiles [0, n_kv) it needs.  Order: L2 sections
// of (b, KV head) groups as in the dK/dV pass; inside a section Q tiles are
// outer (causal: the last, longest, first), then the groups, then the group's
// query heads, so consecutive CTAs share K and V.
struct DqWork {
    int b, g, hq, q0, n_kv;
    int nq, nk, off, qb, kb, vbase;  // as in BwdWork
};

__device__ __forceinline__ DqWork dq_work(const BwdParams& p, unsigned idx) {
    DqWork w;
    const int n_qt = (p.Nq + kBT - 1) / kBT;
    const unsigned all = (unsigned)(p.B * p.Hkv);
    const unsigned S = (unsigned)p.sec_groups;
    const unsigned per_sec = S * (unsigned)p.group * (unsigned)n_qt;
    const unsigned sec = idx / per_sec;
    const unsigned r = idx - sec * per_sec;
    const unsigned rest = all - sec * S;
    const unsigned gs = rest < S ? rest : S;
    const unsigned per_rank = gs * (unsigned)p.group;
    const int rank = (int)(r / per_rank);
    const unsigned rem = r - (unsigned)rank * per_rank;
    const int gl = (int)(rem / (unsigned)p.group);
    const int hl = (int)(rem - (unsigned)gl * (unsigned)p.group);
    const int bg = (int)(sec * S) + gl;
    w.b = bg / p.Hkv;
    w.g = bg - w.b * p.Hkv;
    w.hq = w.g * p.group + hl;
    const int qt = p.causal ? n_qt - 1 - rank : rank;
    w.q0 = qt * kBT;
    if (p.causal) {
        const int last_row = (w.q0 + kBT - 1 < p.Nq - 1 ? w.q0 + kBT - 1 : p.Nq - 1);
        const int last_key = last_row + p.off;
        const int n = last_key < 0 ? 0 : last_key / kBT + 1;
        w.n_kv = n < p.n_kt ? n : p.n_kt;
    } else {
        w.n_kv = p.n_kt;
    }
    w.nq = p.Nq;
    w.nk = p.Nk;
    w.off = p.off;
    w.qb = w.kb = w.vbase = 0;
    return w;
}

// The same for packed batches: item index = (b * Hq + hq) * n_qt + qt, n_qt
// for the longest query length; Q tiles past a sequence's end, and every tile of a
// sequence whose offsets fail the checks, have no work and write nothing.
__device__ __forceinline__ DqWork dq_work_varlen(const BwdParams& p, unsigned idx, unsigned int* err) {
    DqWork w;
    const int n_qt = (p.Nq + kBT - 1) / kBT;
    const int per_b = p.Hq * n_qt;
    w.b = (int)idx / per_b;
    const int rem = (int)idx - w.b * per_b;
    w.hq = rem / n_qt;
    w.g = w.hq / p.group;
    w.q0 = (rem - w.hq * n_qt) * kBT;
    int q0, nq, k0, nk;
    if (!bwd_varlen_seq(p, w.b, q0, nq, k0, nk)) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadSeqlen);
        q0 = nq = k0 = nk = 0;
    }
    w.nq = nq;
    w.nk = nk;
    w.off = nk - nq;
    w.qb = q0;
    w.kb = k0;
    w.vbase = varlen_vbase(q0, w.b);
    const int n_kt = (nk + kBT - 1) / kBT;
    if (w.q0 >= nq) {
        w.n_kv = 0;
    } else if (p.causal) {
        const int last_row = (w.q0 + kBT - 1 < nq - 1 ? w.q0 + kBT - 1 : nq - 1);
        const int last_key = last_row + w.off;
        const int n = last_key < 0 ? 0 : last_key / kBT + 1;
        w.n_kv = n < n_kt ? n : n_kt;
    } else {
        w.n_kv = n_kt;
    }
    return w;
}

// The dQ pass runs a persistent grid as the dK/dV pass does: CTA c takes items
// c, c + gridDim.x, ... of the order above, each one Q tile.
template <bool VARLEN>
__device__ __forceinline__ DqWork dq_item(const BwdParams& p, unsigned idx, unsigned int* err) {
    if constexpr (VARLEN) return dq_work_varlen(p, idx, err);
    else return dq_work(p, idx);
}

template <int D, bool VARLEN>
__device__ void dq_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                            const CUtensorMap* tdo, uint8_t* smem, DqBars* bars, const BwdParams& p,
                            unsigned n_items, unsigned int* err) {
    using C = DqCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    bool ok = true;
    int q_uses = 0;      // Q / dO loads issued (items with work)
    int nk = 0, nv = 0;  // K and V loads issued, over the CTA's items
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const DqWork w = dq_item<VARLEN>(p, idx, err);
        if (w.n_kv == 0) continue;
        // Q and dO of the item, once the previous item's last S and dP have
        // read theirs
        if (q_uses > 0)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->q_empty), (q_uses - 1) & 1, abort_flag));
        if (!ok) break;
        const int bh = w.b * p.Hq + w.hq;
        // K/V head: an index into [B * Hkv], or into [Hkv] of the packed rows
        const int kvh = VARLEN ? w.g : w.b * p.Hkv + w.g;
        if (leader) {
            const uint32_t bar = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(bar, 2 * C::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                if constexpr (VARLEN) {
                    const int r = kRaggedWindow - w.nq + w.q0;
                    tma_load_5d(smem_u32(smem + C::kQ) + c * 16384, tq, bar, 64 * c, w.hq, r, w.qb + w.nq,
                                kRaggedWindow);
                    tma_load_5d(smem_u32(smem + C::kDO) + c * 16384, tdo, bar, 64 * c, w.hq, r, w.qb + w.nq,
                                kRaggedWindow);
                } else {
                    tma_load_3d(smem_u32(smem + C::kQ) + c * 16384, tq, bar, 64 * c, w.q0, bh);
                    tma_load_3d(smem_u32(smem + C::kDO) + c * 16384, tdo, bar, 64 * c, w.q0, bh);
                }
            }
        }
        __syncwarp();
        ++q_uses;
        // K_j into stage (K tile count) % 3 (free once the dQ product three K
        // tiles back has read it), V_j into stage (V tile count) % 2 (free once
        // the dP product two V tiles back has read it).
        for (int j = 0; j < w.n_kv && ok; ++j) {
            const int sk = nk % 3, sv = nv & 1;
            if (nk >= 3)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->k_empty[sk]), ((nk / 3) - 1) & 1,
                                                       abort_flag));
            if (!ok) break;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->k_full[sk]);
                mbar_arrive_expect_tx(bar, C::kTile);
                const uint32_t dst = smem_u32(smem + C::kKRing + sk * C::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if constexpr (VARLEN)
                        tma_load_5d(dst + c * 16384, tk, bar, 64 * c, kvh, kRaggedWindow - w.nk + j * kBT,
                                    w.kb + w.nk, kRaggedWindow);
                    else
                        tma_load_3d(dst + c * 16384, tk, bar, 64 * c, j * kBT, kvh);
                }
            }
            __syncwarp();
            ++nk;
            if (nv >= 2)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->v_empty[sv]), ((nv >> 1) - 1) & 1,
                                                       abort_flag));
            if (!ok) break;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->v_full[sv]);
                mbar_arrive_expect_tx(bar, C::kTile);
                const uint32_t dst = smem_u32(smem + C::kVRing + sv * C::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if constexpr (VARLEN)
                        tma_load_5d(dst + c * 16384, tv, bar, 64 * c, kvh, kRaggedWindow - w.nk + j * kBT,
                                    w.kb + w.nk, kRaggedWindow);
                    else
                        tma_load_3d(dst + c * 16384, tv, bar, 64 * c, j * kBT, kvh);
                }
            }
            __syncwarp();
            ++nv;
        }
    }
    if (!ok && leader) atomicOr(err, kErrTimeout), *((volatile int*)&bars->abort) = 1;
    // Drain: every issued copy lands before the CTA may exit.
    if (q_uses > 0) mbar_wait(smem_u32(&bars->q_full), (q_uses - 1) & 1, nullptr);
    for (int sk = 0; sk < 3 && sk < nk; ++sk) {
        const int uses = (nk - sk + 2) / 3;
        mbar_wait(smem_u32(&bars->k_full[sk]), (uses - 1) & 1, nullptr);
    }
    for (int sv = 0; sv < 2 && sv < nv; ++sv) {
        const int uses = (nv - sv + 1) / 2;
        mbar_wait(smem_u32(&bars->v_full[sv]), (uses - 1) & 1, nullptr);
    }
    __syncwarp();
}

template <int D, bool VARLEN>
__device__ void dq_mma(uint8_t* smem, DqBars* bars, uint32_t tmem, const BwdParams& p, unsigned n_items,
                       unsigned int* err) {
    using C = DqCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idS = make_idesc_bf16(128, 128, 0, 0);
    const uint32_t idQ = make_idesc_bf16(128, D, 0, 1);
    const uint32_t tdP = tmem + 128, tdQ = tmem + 256;
    // K/V tiles are counted over the CTA's items (t): S buffer t & 1, K stage
    // t % 3, V stage t % 2
    auto tS = [&](int t) { return tmem + ((t & 1) ? 384u : 0u); };
    const uint32_t q_k = sdesc_lo(smem_u32(smem + C::kQ), 16);
    const uint32_t do_k = sdesc_lo(smem_u32(smem + C::kDO), 16);
    auto k_k = [&](int sk) { return sdesc_lo(smem_u32(smem + C::kKRing + sk * C::kTile), 16); };
    auto k_mn = [&](int sk) { return sdesc_lo(smem_u32(smem + C::kKRing + sk * C::kTile), 16384); };
    auto v_k = [&](int sv) { return sdesc_lo(smem_u32(smem + C::kVRing + sv * C::kTile), 16); };
    auto wait_all = [&](uint32_t bar, uint32_t parity, int polls) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, polls));
    };
    auto issue_s = [&](int t) {  // S = Q K^T of K/V tile t into buffer t & 1
        if (!wait_all(smem_u32(&bars->k_full[t % 3]), (uint32_t)((t / 3) & 1), 0)) return false;
        tc_fence_after();
        issue_kmajor<D>(tS(t), q_k, k_k(t % 3), idS);
        mma_commit_warp(smem_u32(&bars->s_full[t & 1]));
        return true;
    };
    auto issue_dp = [&](int t) {  // dP = dO V^T of K/V tile t
        if (!wait_all(smem_u32(&bars->v_full[t & 1]), (uint32_t)((t >> 1) & 1), 0)) return false;
        tc_fence_after();
        issue_kmajor<D>(tdP, do_k, v_k(t & 1), idS);
        mma_commit_warp(smem_u32(&bars->v_empty[t & 1]));  // V of tile t is read
        mma_commit_warp(smem_u32(&bars->dp_full));
        return true;
    };
    // Per item: S_0, dP_0, S_1; then per tile j, once dS_j is in TMEM: dQ +=
    // dS_j K_j, dP_{j+1} (into the dP columns the dS warps have read), S_{j+2}
    // (into the buffer dQ_j has read; one CTA's MMAs run in issue order).  The
    // dS warps' exponentials for tile j+1 overlap dQ_j and dP_{j+1}.  An item's
    // first S and dP use columns the previous item's products have read; its
    // first dQ (accumulate = 0) waits for its first dS, which the dS warps
    // write after reading out the previous item's dQ.
    bool ok = true;
    int t0 = 0;  // K/V tiles before this item
    int u = 0;   // items with work
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const DqWork w = dq_item<VARLEN>(p, idx, err);
        const int n = w.n_kv;
        if (n == 0) continue;
        ok = wait_all(smem_u32(&bars->q_full), u & 1, 0);
        if (ok) ok = issue_s(t0);
        if (ok) ok = issue_dp(t0);
        if (ok && n == 1) mma_commit_warp(smem_u32(&bars->q_empty));  // Q and dO are read
        if (ok && n > 1) ok = issue_s(t0 + 1);
        for (int j = 0; j < n && ok; ++j) {
            const int t = t0 + j;
            ok = wait_all(smem_u32(&bars->ds_full), t & 1, 32);
            if (!ok) break;
            tc_fence_after();
            issue_tmem_a(tdQ, tS(t), k_mn(t % 3), idQ, j > 0);  // dQ += dS_j K_j
            mma_commit_warp(smem_u32(&bars->k_empty[t % 3]));   // K_j is read (S_j, dQ_j)
            if (j + 1 < n) {
                if (!(ok = issue_dp(t + 1))) break;
                if (j + 2 == n) mma_commit_warp(smem_u32(&bars->q_empty));  // the last S and dP
            }
            if (j + 2 < n && !(ok = issue_s(t + 2))) break;
        }
        if (ok) mma_commit_warp(smem_u32(&bars->dq_full));
        t0 += n;
        ++u;
    }
    if (!ok && leader) atomicOr(err, kErrTimeout), *((volatile int*)&bars->abort) = 1;
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// P = 2^(S c - lse2) for 32 key columns [kc, kc + 32) of this thread's query
// row (fp32).  lim: key column kc + x is allowed iff kc + x <= lim (causal).
template <bool MASKED>
__device__ __forceinline__ void p_row_chunk(const uint32_t (&s)[32], uint64_t c2, uint64_t nl2,
                                            int kc, int lim, float (&pf)[32]) {
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        const int col = kc + 2 * x;
        float a0, a1;
        f2_split(f2_fma(f2(__uint_as_float(s[2 * x]), __uint_as_float(s[2 * x + 1])), c2, nl2), a0, a1);
        float p0 = ex2(a0), p1 = ex2(a1);
        if constexpr (MASKED) {
            p0 = col <= lim ? p0 : 0.f;
            p1 = col + 1 <= lim ? p1 : 0.f;
        }
        pf[2 * x] = p0;
        pf[2 * x + 1] = p1;
    }
}

// dS = P o (dP - D) for the same 32 columns, packed to bf16 pairs.
__device__ __forceinline__ void ds_row_chunk(const float (&pf)[32], const uint32_t (&dp)[32],
                                             uint64_t nd2, uint32_t (&dd)[16]) {
#pragma unroll
    for (int x = 0; x < 16; ++x) {
        float d0, d1;
        f2_split(f2_mul(f2(pf[2 * x], pf[2 * x + 1]),
                        f2_add(f2(__uint_as_float(dp[2 * x]), __uint_as_float(dp[2 * x + 1])), nd2)),
                 d0, d1);
        dd[x] = pack_bf16x2(d0, d1);
    }
}

template <int D, bool OUT_F32, bool VARLEN>
__device__ void dq_ds(int wq, int grp, int lane, DqBars* bars, uint32_t tmem, const BwdParams& p,
                      unsigned n_items, unsigned int* err) {
    const volatile int* abort_flag = &bars->abort;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tdP = tmem + 128 + lane_off;
    const uint64_t c2 = f2(p.c, p.c);
    bool ok = true;
    int t0 = 0;  // K/V tiles before this item, over the CTA's items
    int u = 0;   // items with work
    for (unsigned idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
        const DqWork w = dq_item<VARLEN>(p, idx, err);
        const int row = w.q0 + wq * 32 + lane;
        const size_t bh = (size_t)w.b * p.Hq + w.hq;
        const size_t vrow = VARLEN ? (size_t)w.hq * p.vstride + (size_t)(w.vbase + row)
                                   : bh * p.Nq_pad + row;
        // +inf past the last query: P = 0 (a tile with no work reads nothing:
        // its rows may lie past the sequence's rows of lse2 / dvec)
        const float lse2 = w.n_kv > 0 ? p.lse2[vrow] : INFINITY;
        const float dval = w.n_kv > 0 ? p.dvec[vrow] : 0.f;
        const uint64_t nl2 = f2(-lse2, -lse2), nd2 = f2(-dval, -dval);
        for (int j = 0; j < w.n_kv && ok; ++j) {
            const int t = t0 + j;
            const uint32_t tS = tmem + ((t & 1) ? 384u : 0u) + lane_off;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->s_full[t & 1]), (t >> 1) & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            const int lim = row + w.off - j * kBT;  // causal: key column c allowed iff c <= lim
            const bool masked = __any_sync(0xFFFFFFFFu, p.causal && lim < kBT - 1);
            // Phase 1: P from S for this warpgroup's 64 key columns (needs S_j
            // only; runs while dQ_{j-1} and dP_j compute)
            float pf0[32], pf1[32];
            auto phase1 = [&](int cc, float (&pf)[32]) {
                uint32_t sv[32];
                tmem_ld32(tS + cc * 32, sv);
                tmem_wait_ld();
                if (masked)
                    p_row_chunk<true>(sv, c2, nl2, cc * 32, p.causal ? lim : kBT, pf);
                else
                    p_row_chunk<false>(sv, c2, nl2, cc * 32, kBT, pf);
            };
            phase1(2 * grp, pf0);
            phase1(2 * grp + 1, pf1);
            // Phase 2: dS from P and dP, as bf16 over the S columns this
            // warpgroup read
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->dp_full), t & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            auto phase2 = [&](int cc, const float (&pf)[32]) {
                uint32_t dp[32], dd[16];
                tmem_ld32(tdP + cc * 32, dp);
                tmem_wait_ld();
                ds_row_chunk(pf, dp, nd2, dd);
                tmem_st16(tS + a_chunk_col(cc), dd);
            };
            phase2(2 * grp, pf0);
            phase2(2 * grp + 1, pf1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->ds_full));
        }
        if (!ok) break;
        if (w.n_kv > 0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->dq_full), u & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
        }
        // every lane runs the (warp-collective) TMEM loads; rows past Nq store
        // nothing.  This warp's first query row and how many of its rows are
        // inside Nq (packed batches: rows of Hq * d elements, the head's d
        // columns at hq * d).  The next item's first dQ product (accumulate =
        // 0) is issued only after this warpgroup's next dS arrival, which
        // follows these reads.
        const size_t wrow0 = VARLEN ? (size_t)(w.qb + w.q0 + wq * 32) : bh * p.Nq + (size_t)(w.q0 + wq * 32);
        const int rows_live = w.nq - (w.q0 + wq * 32);
        const size_t row_elems = VARLEN ? (size_t)p.Hq * p.d_act : (size_t)p.d_act;
        void* dq_base = static_cast<uint8_t*>(p.dq) + (VARLEN ? (size_t)w.hq * p.d_act * (OUT_F32 ? 4 : 2) : 0);
#pragma unroll 1
        for (int cc = grp * (D / 2); cc < (grp + 1) * (D / 2); cc += 32) {  // this warpgroup's half
            float v[32];
            if (w.n_kv > 0) {
                uint32_t r[32];
                tmem_ld32(tmem + 256 + cc + lane_off, r);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]) * p.scale;
            } else {
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] = 0.f;
            }
            const int nc = p.d_act - cc < 32 ? p.d_act - cc : 32;
            if (nc > 0) store_rows32_pairs<OUT_F32>(dq_base, wrow0, row_elems, cc, v, nc, rows_live, lane);
        }
        if (w.n_kv > 0) {
            tc_fence_before();
            t0 += w.n_kv;
            ++u;
        }
    }
    if (!ok) {
        atomicOr(err, kErrTimeout);
        *((volatile int*)&bars->abort) = 1;
    }
}

template <int D, bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreadsEw, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const BwdParams p, unsigned int* err) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
    if ((uintptr_t)(smem - smem_raw) + C::kLayout > (uintptr_t)C::kSmemBytes) {
        if (threadIdx.x == 0) atomicOr(err, kErrLayout);
        return;
    }
    DqBars* bars = reinterpret_cast<DqBars*>(smem + C::kBar);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned n_items = (unsigned)(p.B * p.Hq * ((p.Nq + kBT - 1) / kBT));
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_empty), 1);  // the commit after an item's last S and dP
        for (int s = 0; s < 3; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
            mbar_init(smem_u32(&bars->s_full[s]), 1);
        }
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->ds_full), 8);
        mbar_init(smem_u32(&bars->dq_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (warp == 0) dq_producer<D, VARLEN>(&tq, &tk, &tv, &tdo, smem, bars, p, n_items, err);
    else if (warp == 1) dq_mma<D, VARLEN>(smem, bars, tmem, p, n_items, err);
    else if (warp >= 4) dq_ds<D, OUT_F32, VARLEN>(warp & 3, (warp - 4) >> 2, lane, bars, tmem, p, n_items, err);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
// D = dO . O and lse2 = LSE log2(e) for every padded query row (padding: 0
// and +inf).  LPR lanes share a row, each reading 8 consecutive elements of
// dO and of O per 16-byte load (rows start on 16-byte boundaries: d % 8 == 0
// and both arrays 16-byte aligned), so a warp covers 32 / LPR rows with
// whole-sector loads; their partial sums meet by shuffles inside the group.
template <int LPR>
__global__ void __launch_bounds__(256)
attn_bwd_prep_kernel(const void* __restrict__ o, int o_f32, const __nv_bfloat16* __restrict__ dout,
                     const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ dvec,
                     long long rows_pad, int Nq, int Nq_pad, int dh) {
    constexpr int kRowsPerWarp = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const long long r = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRowsPerWarp + lane / LPR;
    const bool live_row = r < rows_pad;
    const long long bh = live_row ? r / Nq_pad : 0;
    const int i = live_row ? (int)(r - bh * Nq_pad) : Nq;
    float sum = 0.f;
    if (i < Nq) {
        const size_t base = ((size_t)bh * Nq + i) * dh;
        for (int c = sub * 8; c < dh; c += LPR * 8) {
            const uint4 g = *reinterpret_cast<const uint4*>(dout + base + c);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            float ov[8];
            if (o_f32) {
                const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + c);
                const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + c + 4);
                ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
                ov[4] = b.x; ov[5] = b.y; ov[6] = b.z; ov[7] = b.w;
            } else {
                const uint4 h = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o) + base + c);
                const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ov[2 * e] = __uint_as_float(hw[e] << 16);
                    ov[2 * e + 1] = __uint_as_float(hw[e] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sum = fmaf(__uint_as_float(gw[e] << 16), ov[2 * e], sum);
                sum = fmaf(__uint_as_float(gw[e] & 0xFFFF0000u), ov[2 * e + 1], sum);
            }
        }
    }
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, s);
    if (live_row && sub == 0) {
        dvec[r] = i < Nq ? sum : 0.f;
        lse2[r] = i < Nq ? lse[(size_t)bh * Nq + i] * kBwdLog2e : INFINITY;
    }
}

// The same for packed batches: block (b, hq, chunk) covers rows
// [chunk * rows, (chunk + 1) * rows) of sequence b's rows padded to whole
// 128-row tiles, in the varlen_vbase layout; rows past the sequence's queries
// get lse2 = +inf, D = 0.  A sequence whose offsets leave the arrays is
// skipped here (the passes report it and compute nothing for it).
template <int LPR>
__global__ void __launch_bounds__(256)
attn_bwd_prep_varlen_kernel(const void* __restrict__ o, int o_f32, const __nv_bfloat16* __restrict__ dout,
                            const float* __restrict__ lse, float* __restrict__ lse2,
                            float* __restrict__ dvec, const int* __restrict__ cu_q, int Hq,
                            int total_q, int vstride, int chunks, int dh) {
    constexpr int kRowsPerWarp = 32 / LPR;
    constexpr int kRowsPerBlock = 8 * kRowsPerWarp;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const int per_b = Hq * chunks;
    const int b = (int)blockIdx.x / per_b;
    const int rem = (int)blockIdx.x - b * per_b;
    const int hq = rem / chunks;
    const int i = (rem - hq * chunks) * kRowsPerBlock + (threadIdx.x >> 5) * kRowsPerWarp + lane / LPR;
    const int q0 = __ldg(cu_q + b), qe = __ldg(cu_q + b + 1);
    const int nq = qe - q0;
    const bool seq_ok = 0 <= q0 && q0 <= qe && qe <= total_q;
    const bool live_row = seq_ok && i < (nq + kBT - 1) / kBT * kBT;
    const bool valid = live_row && i < nq;
    float sum = 0.f;
    if (valid) {
        const size_t base = ((size_t)(q0 + i) * Hq + hq) * dh;
        for (int c = sub * 8; c < dh; c += LPR * 8) {
            const uint4 g = *reinterpret_cast<const uint4*>(dout + base + c);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            float ov[8];
            if (o_f32) {
                const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + c);
                const float4 bb = *reinterpret_cast<const float4*>(static_cast<const float*>(o) + base + c + 4);
                ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
                ov[4] = bb.x; ov[5] = bb.y; ov[6] = bb.z; ov[7] = bb.w;
            } else {
                const uint4 h = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o) + base + c);
                const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ov[2 * e] = __uint_as_float(hw[e] << 16);
                    ov[2 * e + 1] = __uint_as_float(hw[e] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sum = fmaf(__uint_as_float(gw[e] << 16), ov[2 * e], sum);
                sum = fmaf(__uint_as_float(gw[e] & 0xFFFF0000u), ov[2 * e + 1], sum);
            }
        }
    }
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, s);
    if (live_row && sub == 0) {
        const size_t r = (size_t)hq * vstride + (size_t)(varlen_vbase(q0, b) + i);
        dvec[r] = valid ? sum : 0.f;
        lse2[r] = valid ? lse[(size_t)hq * total_q + (size_t)(q0 + i)] * kBwdLog2e : INFINITY;
    }
}

attn_status_t launch_bwd_prep_varlen(const void* o, int o_f32, const void* dout, const float* lse,
                                     float* lse2, float* dvec, const BwdParams& p, cudaStream_t stream) {
    const auto* g = static_cast<const __nv_bfloat16*>(dout);
    const int dh = p.d_act;
    const int lpr = dh <= 64 ? 8 : dh <= 128 ? 16 : 32;
    const int rows_per_block = 8 * (32 / lpr);
    const int rows_pad = (p.Nq + kBT - 1) / kBT * kBT;
    const int chunks = (rows_pad + rows_per_block - 1) / rows_per_block;
    const long long grid = (long long)p.B * p.Hq * chunks;
    if (grid >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
#define GB300_PREP_VARLEN(L)                                                                       \
    attn_bwd_prep_varlen_kernel<L><<<(unsigned)grid, 256, 0, stream>>>(o, o_f32, g, lse, lse2, dvec, \
                                                                       p.cu_q, p.Hq, p.total_q,      \
                                                                       p.vstride, chunks, dh)
    if (lpr == 8) GB300_PREP_VARLEN(8);
    else if (lpr == 16) GB300_PREP_VARLEN(16);
    else GB300_PREP_VARLEN(32);
#undef GB300_PREP_VARLEN
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// The prep launch for head dim dh (<= 256): 8, 16 or 32 lanes per row.
attn_status_t launch_bwd_prep(const void* o, int o_f32, const void* dout, const float* lse,
                              float* lse2, float* dvec, long long rows_pad, int Nq, int Nq_pad,
                              int dh, cudaStream_t stream) {
    const auto* g = static_cast<const __nv_bfloat16*>(dout);
    const int lpr = dh <= 64 ? 8 : dh <= 128 ? 16 : 32;
    const long long rows_per_block = 8ll * (32 / lpr);
    const unsigned grid = (unsigned)((rows_pad + rows_per_block - 1) / rows_per_block);
    if (lpr == 8)
        attn_bwd_prep_kernel<8><<<grid, 256, 0, stream>>>(o, o_f32, g, lse, lse2, dvec, rows_pad, Nq, Nq_pad, dh);
    else if (lpr == 16)
        attn_bwd_prep_kernel<16><<<grid, 256, 0, stream>>>(o, o_f32, g, lse, lse2, dvec, rows_pad, Nq, Nq_pad, dh);
    else
        attn_bwd_prep_kernel<32><<<grid, 256, 0, stream>>>(o, o_f32, g, lse, lse2, dvec, rows_pad, Nq, Nq_pad, dh);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, bool OUT_F32, bool VARLEN = false>
attn_status_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                           const BwdParams& p, const void* o, int o_f32,
                           const void* dout, const float* lse, float* lse2, float* dvec,
                           cudaStream_t stream, const DeviceInfo& dev) {
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 BwdCfg<D>::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_dq_kernel<D, OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DqCfg<D>::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    attn_status_t st;
    if constexpr (VARLEN) {
        st = launch_bwd_prep_varlen(o, o_f32, dout, lse, lse2, dvec, p, stream);
    } else {
        const long long rows_pad = (long long)p.B * p.Hq * p.Nq_pad;
        st = launch_bwd_prep(o, o_f32, dout, lse, lse2, dvec, rows_pad, p.Nq, p.Nq_pad, p.d_act, stream);
    }
    if (st != ATTN_OK) return st;
    // (packed batches: units at the longest lengths; the tiles past a
    // sequence's end have no work).  The dK/dV pass is persistent: at most one
    // CTA per SM, each taking every gridDim.x-th key tile.
    const long long kv_items = (long long)p.B * p.Hkv * p.n_kt;
    const long long kv_ctas = kv_items < dev.num_sms ? kv_items : dev.num_sms;
    attn_bwd_dkdv_kernel<D, OUT_F32, VARLEN><<<(unsigned)kv_ctas, kBwdThreadsEw, BwdCfg<D>::kSmemBytes,
                                               stream>>>(tq, tk, tv, tdo, tdk, tdv, p, dev.err_word);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    const long long q_items = (long long)p.B * p.Hq * ((p.Nq + kBT - 1) / kBT);
    const long long q_ctas = q_items < dev.num_sms ? q_items : dev.num_sms;  // persistent, as above
    attn_bwd_dq_kernel<D, OUT_F32, VARLEN><<<(unsigned)q_ctas, kBwdThreadsEw, DqCfg<D>::kSmemBytes,
                                             stream>>>(tq, tk, tv, tdo, p, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Head dims 128 < d <= 256 (kernels built for 256 columns; columns past d are
// zeros in every tile and are not written).
//
// At d = 256 the dK/dV pass's accumulators alone (dV and dK, 256 columns
// each) fill TMEM, and a 128-row Q or dO tile is 64 KiB, so these kernels use
// other tile shapes, each product a shape the d > 128 forward also runs:
//  dkdv  one CTA per (b, KV head g, 128-key tile, column half h of d).  K and
//        V of the tile stay in shared memory (64 KiB each); Q (with its lse2
//        and D rows) streams in 64-row tiles through two buffers, dO through
//        one.  Per Q tile:
//          S^T = K Q^T, dP^T = V dO^T           (M=128, N=64, K=256)
//          P^T, dS^T as in the d <= 128 pass    (64 query columns per key row)
//          dV_h += P^T dO_h, dK_h += dS^T Q_h   (M=128, N=128, K=64: columns
//                                                 [128h, 128h + 128) of d)
//        S^T and dP^T are computed by both CTAs of a key tile (the two
//        halves), so the pass does 3 of its 4 products' work twice.
//        TMEM: S^T [0,64) (P^T over [0,32)), dP^T [64,128) (dS^T over
//        [64,96)), dV_h [128,256), dK_h [256,384).
//  dq    one CTA per (b, query head, 128-row Q tile).  Q and dO stay in
//        shared memory; K streams in 64-key tiles through two buffers, V
//        through one.  Per K/V tile: S = Q K^T, dP = dO V^T (M=128, N=64,
//        K=256), dS as in the d <= 128 pass, dQ += dS K (M=128, N=256, K=64).
//        TMEM: S in [0,64) for even K/V tiles and [64,128) for odd ones (dS
//        over its first 32 columns), dP [128,192), dQ [192,448).
// Both passes issue the next tile's first product while the elementwise warps
// work on the current tile (the dK/dV pass S^T(i+1) after dV(i), the dQ pass
// S_{j+2} after dQ_j).  Packed batches (VARLEN) use the d <= 128 passes' work
// decoding with the Q (dK/dV) and K/V (dQ) tiles read through ragged tensor
// maps with 64-row boxes.
// ---------------------------------------------------------------------------
constexpr int kWD = 256;    // tile columns
constexpr int kWQ = 64;     // query rows per dkdv Q tile, keys per dq K/V tile
constexpr uint32_t kWBwdDescHi = sdesc_hi_sw128(1024);

// dkdv: K, V resident | Q in two buffers (with lse2[64], D[64] each) | dO
struct WideDkdvCfg {
    static constexpr int kBig = kBT * kWD * 2;     // 128 rows x 256: 4 chunks of 16 KiB
    static constexpr int kSmall = kWQ * kWD * 2;   // 64 rows x 256: 4 chunks of 8 KiB
    static constexpr int kK = 0;
    static constexpr int kV = kBig;
    static constexpr int kQ = 2 * kBig;                 // 2 buffers
    static constexpr int kDO = 2 * kBig + 2 * kSmall;   // 1 buffer
    static constexpr int kLD = 2 * kBig + 3 * kSmall;   // 2 x (lse2[64], D[64])
    static constexpr int kBar = kLD + 1024;
    static constexpr int kLayout = kBar + 256;
    static constexpr int kSmemBytes = kLayout + 1024;
    static_assert(kSmemBytes <= kMaxSmemPerBlock, "shared memory budget");
};

struct __align__(8) WideDkdvBars {
    uint64_t kv_full;
    uint64_t q_full[2], q_empty[2];  // Q_i and its lse2 / D rows, buffer i & 1
    uint64_t do_full, do_empty;      // dO_i
    uint64_t s_full, dp_full, p_full, ds_full, acc_full, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(WideDkdvBars) <= 256, "barrier block");

// dq: Q, dO resident | K in two buffers | V
struct WideDqCfg {
    static constexpr int kBig = kBT * kWD * 2;     // 128 rows x 256: 4 chunks of 16 KiB
    static constexpr int kSmall = kWQ * kWD * 2;   // 64 rows x 256: 4 chunks of 8 KiB
    static constexpr int kQ = 0;
    static constexpr int kDO = kBig;
    static constexpr int kK = 2 * kBig;                 // 2 buffers
    static constexpr int kV = 2 * kBig + 2 * kSmall;    // 1 buffer
    static constexpr int kBar = 2 * kBig + 3 * kSmall;
    static constexpr int kLayout = kBar + 256;
    static constexpr int kSmemBytes = kLayout + 1024;
    static_assert(kSmemBytes <= kMaxSmemPerBlock, "shared memory budget");
};

struct __align__(8) WideDqBars {
    uint64_t res_full;                 // Q, dO
    uint64_t k_full[2], k_empty[2];    // K_j, buffer j & 1
    uint64_t v_full, v_empty;          // V_j
    uint64_t s_full[2];                // S_j, TMEM buffer j & 1
    uint64_t dp_full, ds_full, acc_full, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(WideDqBars) <= 256, "barrier block");

// S = A B^T with M = 128, N = 64, K = 256: A 128 rows K-major (chunks of 64
// columns 16 KiB apart), B 64 rows K-major (chunks 8 KiB apart).
__device__ __forceinline__ void wbwd_issue_s(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < kWD / 16; ++kk) {
        const uint32_t in = (kk & 3) * (32 >> 4);
        mma_ss_warp(d_tmem, sdesc_join(a_lo + (kk >> 2) * ((kBT * 128) >> 4) + in, kWBwdDescHi),
                    sdesc_join(b_lo + (kk >> 2) * ((kWQ * 128) >> 4) + in, kWBwdDescHi), idesc,
                    kk > 0 ? 1u : 0u);
    }
}

// D += A B with A from TMEM (bf16 pairs, 8 columns per 16 rows of K, K = 64)
// and B a 64-row tile MN-major (LBO 8 KiB between 64-column chunks, 16 rows =
// 2 KiB per K step); N per idesc.
__device__ __forceinline__ void wbwd_issue_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                              uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kWQ / 16; ++kk)
        mma_ts_warp(d_tmem, a_tmem + kk * 8, sdesc_join(b_lo + kk * (2048 >> 4), kWBwdDescHi), idesc,
                    (accumulate || kk > 0) ? 1u : 0u);
}

struct WideDkdvWork {
    int b, g, kt, k0, half, qt_first, n_qt_cta, n_tiles;
    int nq, nk, off, qb, kb, vbase;  // as in BwdWork
};

// CTA index -> (column half, then the dkdv pass's section order of key tiles).
__device__ __forceinline__ WideDkdvWork wide_dkdv_work(const BwdParams& p) {
    WideDkdvWork w;
    const unsigned idx = blockIdx.x >> 1;
    w.half = (int)(blockIdx.x & 1u);
    const unsigned all = (unsigned)(p.B * p.Hkv);
    const unsigned S = (unsigned)p.sec_groups;
    const unsigned per_sec = S * (unsigned)p.n_kt;
    const unsigned sec = idx / per_sec;
    const unsigned r = idx - sec * per_sec;
    const unsigned rest = all - sec * S;
    const unsigned gs = rest < S ? rest : S;
    w.kt = (int)(r / gs);
    const int bg = (int)(sec * S + (r - (unsigned)w.kt * gs));
    w.b = bg / p.Hkv;
    w.g = bg - w.b * p.Hkv;
    w.k0 = w.kt * kBT;
    const int n_qt = (p.Nq + kWQ - 1) / kWQ;
    int first = 0;
    if (p.causal) {
        const int lo = w.k0 - p.off;  // the first query that sees key k0
        first = lo <= 0 ? 0 : lo / kWQ;
    }
    w.qt_first = first;
    w.n_qt_cta = n_qt - first > 0 ? n_qt - first : 0;
    w.n_tiles = w.n_qt_cta * p.group;
    w.nq = p.Nq;
    w.nk = p.Nk;
    w.off = p.off;
    w.qb = w.kb = w.vbase = 0;
    return w;
}

// The same for packed batches: CTA index = ((b * Hkv + g) * n_kt + kt) * 2 +
// column half, n_kt for the longest key length; key tiles past a sequence's
// end, and every tile of a sequence whose offsets fail the checks, have no
// work and write nothing.
__device__ __forceinline__ WideDkdvWork wide_dkdv_work_varlen(const BwdParams& p, unsigned int* err) {
    WideDkdvWork w;
    const int idx = (int)(blockIdx.x >> 1);
    w.half = (int)(blockIdx.x & 1u);
    const int per_b = p.Hkv * p.n_kt;
    w.b = idx / per_b;
    const int rem = idx - w.b * per_b;
    w.g = rem / p.n_kt;
    w.kt = rem - w.g * p.n_kt;
    w.k0 = w.kt * kBT;
    int q0, nq, k0, nk;
    if (!bwd_varlen_seq(p, w.b, q0, nq, k0, nk)) {
        if (threadIdx.x == 0) atomicOr(err, kErrBadSeqlen);
        q0 = nq = k0 = nk = 0;
    }
    w.nq = nq;
    w.nk = nk;
    w.off = nk - nq;
    w.qb = q0;
    w.kb = k0;
    w.vbase = varlen_vbase(q0, w.b);
    const int n_qt = (nq + kWQ - 1) / kWQ;
    int first = 0;
    if (p.causal) {
        const int lo = w.k0 - w.off;
        first = lo <= 0 ? 0 : lo / kWQ;
    }
    w.qt_first = first;
    w.n_qt_cta = (w.k0 < nk && n_qt - first > 0) ? n_qt - first : 0;
    w.n_tiles = w.n_qt_cta * p.group;
    return w;
}

template <bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_wide_dkdv_kernel(const __grid_constant__ CUtensorMap tq64, const __grid_constant__ CUtensorMap tdo64,
                          const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                          const BwdParams p, unsigned int* err) {
    using C = WideDkdvCfg;
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
    if ((uintptr_t)(smem - smem_raw) + C::kLayout > (uintptr_t)C::kSmemBytes) {
        if (threadIdx.x == 0) atomicOr(err, kErrLayout);
        return;
    }
    WideDkdvBars* bars = reinterpret_cast<WideDkdvBars*>(smem + C::kBar);
    const volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WideDkdvWork w = VARLEN ? wide_dkdv_work_varlen(p, err) : wide_dkdv_work(p);
    auto raise_abort = [&]() {
        atomicOr(err, kErrTimeout);
        *((volatile int*)&bars->abort) = 1;
    };
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(smem_u32(&bars->q_full[b2]), 1);
            mbar_init(smem_u32(&bars->q_empty[b2]), 1 + 4);  // the dK commit + 4 P/dS warps
        }
        mbar_init(smem_u32(&bars->do_full), 1);
        mbar_init(smem_u32(&bars->do_empty), 1);  // the dV commit (dP^T has read dO before it)
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->p_full), 4);
        mbar_init(smem_u32(&bars->ds_full), 4);
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq64);
        tma_prefetch_desc(&tdo64);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---- producer: K, V once; per 64-row tile Q (+ lse2, D) into buffer i & 1
        // and dO into its one buffer.  Order Q_0, dO_0, Q_1, then dO_i once dV(i-1)
        // has read dO_{i-1}, and Q_{i+1} once dK(i-1) and the P/dS warps are done
        // with buffer (i+1) & 1.
        const bool leader = elect_one();
        const int kvh = VARLEN ? w.g : w.b * p.Hkv + w.g;
        if (leader) {
            const uint32_t bar = smem_u32(&bars->kv_full);
            mbar_arrive_expect_tx(bar, 2 * C::kBig);
#pragma unroll
            for (int c = 0; c < kWD / 64; ++c) {
                if constexpr (VARLEN) {
                    const int r = kRaggedWindow - w.nk + w.k0;
                    tma_load_5d(smem_u32(smem + C::kK) + c * 16384, &tk, bar, 64 * c, kvh, r, w.kb + w.nk,
                                kRaggedWindow);
                    tma_load_5d(smem_u32(smem + C::kV) + c * 16384, &tv, bar, 64 * c, kvh, r, w.kb + w.nk,
                                kRaggedWindow);
                } else {
                    tma_load_3d(smem_u32(smem + C::kK) + c * 16384, &tk, bar, 64 * c, w.k0, kvh);
                    tma_load_3d(smem_u32(smem + C::kV) + c * 16384, &tv, bar, 64 * c, w.k0, kvh);
                }
            }
        }
        __syncwarp();
        // tile i: its first query row, and its head (an index into [B * Hq], or
        // into [Hq] of the packed rows)
        auto tile_rows = [&](int i, int& q0, int& bh) {
            const int hq = w.g * p.group + i / w.n_qt_cta;
            q0 = (w.qt_first + i % w.n_qt_cta) * kWQ;
            bh = VARLEN ? hq : w.b * p.Hq + hq;
        };
        // the 64-row tile of Q or dO at q0 (packed: rows past the sequence's
        // queries read as zeros)
        auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int q0, int bh) {
#pragma unroll
            for (int c = 0; c < kWD / 64; ++c) {
                if constexpr (VARLEN)
                    tma_load_5d(dst + c * 8192, map, bar, 64 * c, bh, kRaggedWindow - w.nq + q0, w.qb + w.nq,
                                kRaggedWindow);
                else
                    tma_load_3d(dst + c * 8192, map, bar, 64 * c, q0, bh);
            }
        };
        bool ok = true;
        int nq = 0, ndo = 0;  // Q and dO tiles issued
        auto load_q = [&](int i) {
            const int qb = i & 1;
            if (i >= 2)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->q_empty[qb]), ((i >> 1) - 1) & 1,
                                                       abort_flag));
            if (!ok) return;
            int q0, bh;
            tile_rows(i, q0, bh);
            if (leader) {
                const uint32_t bar = smem_u32(&bars->q_full[qb]);
                mbar_arrive_expect_tx(bar, C::kSmall + 2 * kWQ * 4);
                load_rows(smem_u32(smem + C::kQ + qb * C::kSmall), &tq64, bar, q0, bh);
                const size_t row = VARLEN ? (size_t)bh * p.vstride + (size_t)(w.vbase + q0)
                                          : (size_t)bh * p.Nq_pad + q0;
                const uint32_t ld = smem_u32(smem + C::kLD + qb * 512);
                bulk_load(ld, p.lse2 + row, kWQ * 4, bar);
                bulk_load(ld + kWQ * 4, p.dvec + row, kWQ * 4, bar);
            }
            __syncwarp();
            ++nq;
        };
        auto load_do = [&](int i) {
            if (i >= 1)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->do_empty), (i - 1) & 1, abort_flag));
            if (!ok) return;
            int q0, bh;
            tile_rows(i, q0, bh);
            if (leader) {
                const uint32_t bar = smem_u32(&bars->do_full);
                mbar_arrive_expect_tx(bar, C::kSmall);
                load_rows(smem_u32(smem + C::kDO), &tdo64, bar, q0, bh);
            }
            __syncwarp();
            ++ndo;
        };
        if (w.n_tiles > 0) {
            load_q(0);
            if (ok) load_do(0);
            if (ok && w.n_tiles > 1) load_q(1);
            for (int i = 1; i < w.n_tiles && ok; ++i) {
                load_do(i);
                if (ok && i + 1 < w.n_tiles) load_q(i + 1);
            }
        }
        if (!ok && leader) raise_abort();
        // Drain: every issued copy lands before the CTA may exit.
        mbar_wait(smem_u32(&bars->kv_full), 0, nullptr);
        for (int qb = 0; qb < 2 && qb < nq; ++qb) {
            const int uses = (nq - qb + 1) / 2;
            mbar_wait(smem_u32(&bars->q_full[qb]), (uses - 1) & 1, nullptr);
        }
        if (ndo > 0) mbar_wait(smem_u32(&bars->do_full), (ndo - 1) & 1, nullptr);
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer.  S^T(0), dP^T(0); per tile i: dV(i) once P^T(i) is in
        // TMEM, then S^T(i+1) into the columns dV(i) has read; dK(i) once dS^T(i)
        // is in TMEM, then dP^T(i+1) into the columns dK(i) has read (one CTA's
        // MMAs run in issue order).  The P/dS warps work on tile i+1's P^T while
        // dK(i) and the load of dO_{i+1} proceed.
        const bool leader = elect_one();
        const uint32_t idS = make_idesc_bf16(128, kWQ, 0, 0);
        const uint32_t idH = make_idesc_bf16(128, 128, 0, 1);
        const uint32_t tS = tmem, tdP = tmem + 64, tdV = tmem + 128, tdK = tmem + 256;
        const uint32_t k_lo = sdesc_lo(smem_u32(smem + C::kK), 16);
        const uint32_t v_lo = sdesc_lo(smem_u32(smem + C::kV), 16);
        const uint32_t do_lo = sdesc_lo(smem_u32(smem + C::kDO), 16);
        // this CTA's column half of Q and dO as MN-major B operands
        const uint32_t do_mn = sdesc_lo(smem_u32(smem + C::kDO) + w.half * 2 * 8192, 8192);
        auto q_lo = [&](int qb) { return sdesc_lo(smem_u32(smem + C::kQ + qb * C::kSmall), 16); };
        auto q_mn = [&](int qb) {
            return sdesc_lo(smem_u32(smem + C::kQ + qb * C::kSmall) + w.half * 2 * 8192, 8192);
        };
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, 32));
        };
        auto issue_st = [&](int i) {  // S^T(i) = K Q_i^T
            if (!wait_all(smem_u32(&bars->q_full[i & 1]), (i >> 1) & 1)) return false;
            tc_fence_after();
            wbwd_issue_s(tS, k_lo, q_lo(i & 1), idS);
            mma_commit_warp(smem_u32(&bars->s_full));
            return true;
        };
        auto issue_dpt = [&](int i) {  // dP^T(i) = V dO_i^T
            if (!wait_all(smem_u32(&bars->do_full), i & 1)) return false;
            tc_fence_after();
            wbwd_issue_s(tdP, v_lo, do_lo, idS);
            mma_commit_warp(smem_u32(&bars->dp_full));
            return true;
        };
        bool ok = true;
        if (w.n_tiles > 0) {
            ok = wait_all(smem_u32(&bars->kv_full), 0);
            if (ok) ok = issue_st(0);
            if (ok) ok = issue_dpt(0);
        }
        for (int i = 0; i < w.n_tiles && ok; ++i) {
            const bool more = i + 1 < w.n_tiles;
            ok = wait_all(smem_u32(&bars->p_full), i & 1);
            if (!ok) break;
            tc_fence_after();
            wbwd_issue_ta(tdV, tS, do_mn, idH, i > 0);             // dV_h += P^T dO_h
            mma_commit_warp(smem_u32(&bars->do_empty));            // dO_i is read
            if (more && !(ok = issue_st(i + 1))) break;
            ok = wait_all(smem_u32(&bars->ds_full), i & 1);
            if (!ok) break;
            tc_fence_after();
            wbwd_issue_ta(tdK, tdP, q_mn(i & 1), idH, i > 0);      // dK_h += dS^T Q_h
            mma_commit_warp(smem_u32(&bars->q_empty[i & 1]));      // Q_i is read
            if (more && !(ok = issue_dpt(i + 1))) break;
        }
        if (ok && w.n_tiles > 0) mma_commit_warp(smem_u32(&bars->acc_full));
        if (!ok && leader) raise_abort();
        mma_commit_warp(smem_u32(&bars->drain));
        mbar_wait(smem_u32(&bars->drain), 0, nullptr);
        __syncwarp();
    } else if (warp >= 4) {
        // ---- P^T / dS^T (one key row per thread), then the dK_h / dV_h epilogue
        const int wq = warp & 3;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off, tdP = tmem + 64 + lane_off;
        const int jg = w.k0 + wq * 32 + lane;
        bool ok = true;
        for (int i = 0; i < w.n_tiles && ok; ++i) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->s_full), i & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            const int q0 = (w.qt_first + i % w.n_qt_cta) * kWQ;
            const int lim = jg - w.off - q0;  // causal: column x allowed iff x >= lim
            const bool masked = p.causal && (q0 + w.off < w.k0 + kBT - 1);
            const uint32_t lse2s = smem_u32(smem + C::kLD + (i & 1) * 512);
            const uint32_t ds_vec = lse2s + kWQ * 4;
            float pf0[32], pf1[32];
            {
                uint32_t sv[32], pp[16];
                tmem_ld32(tS, sv);
                tmem_wait_ld();
                if (masked) p_chunk<true>(sv, lse2s, 0, p.c, lim, pf0, pp);
                else p_chunk<false>(sv, lse2s, 0, p.c, lim, pf0, pp);
                tmem_st16(tS, pp);
                tmem_ld32(tS + 32, sv);
                tmem_wait_ld();
                if (masked) p_chunk<true>(sv, lse2s, 32, p.c, lim, pf1, pp);
                else p_chunk<false>(sv, lse2s, 32, p.c, lim, pf1, pp);
                tmem_st16(tS + 16, pp);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->p_full));
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->dp_full), i & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dp[32], dd[16];
                tmem_ld32(tdP, dp);
                tmem_wait_ld();
                ds_chunk_t(pf0, dp, ds_vec, 0, dd);
                tmem_st16(tdP, dd);
                tmem_ld32(tdP + 32, dp);
                tmem_wait_ld();
                ds_chunk_t(pf1, dp, ds_vec, 32, dd);
                tmem_st16(tdP + 16, dd);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&bars->ds_full));
                mbar_arrive(smem_u32(&bars->q_empty[i & 1]));  // lse2 and D of the tile are read
            }
        }
        if (!ok) {
            raise_abort();
        } else {
            // dK_h = scale dS^T Q_h, dV_h = P^T dO_h: columns [128h, 128h + 128)
            // (packed batches: rows of Hkv * d elements, the head's d columns at g * d)
            const size_t wrow0 = VARLEN ? (size_t)(w.kb + w.k0 + wq * 32)
                                        : ((size_t)w.b * p.Hkv + w.g) * p.Nk + (size_t)(w.k0 + wq * 32);
            const int rows_live = w.nk - (w.k0 + wq * 32);
            const size_t row_elems = VARLEN ? (size_t)p.Hkv * p.d_act : (size_t)p.d_act;
            const size_t head_off = VARLEN ? (size_t)w.g * p.d_act * (OUT_F32 ? 4 : 2) : 0;
            void* dk_base = static_cast<uint8_t*>(p.dk) + head_off;
            void* dv_base = static_cast<uint8_t*>(p.dv) + head_off;
            const int c0 = w.half * 128;
            const bool have = w.n_tiles > 0;
            if (have) {
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->acc_full), 0, abort_flag));
                if (!ok) raise_abort();
                else tc_fence_after();
            }
            if (ok) {
#pragma unroll 1
                for (int cc = 0; cc < 128; cc += 32) {
                    const int nc = p.d_act - (c0 + cc) < 32 ? p.d_act - (c0 + cc) : 32;
                    float v[32];
                    uint32_t r[32];
                    if (have) {
                        tmem_ld32(tmem + 128 + cc + lane_off, r);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = have ? __uint_as_float(r[x]) : 0.f;
                    if (nc > 0) store_rows32_pairs<OUT_F32>(dv_base, wrow0, row_elems, c0 + cc, v, nc, rows_live, lane);
                    if (have) {
                        tmem_ld32(tmem + 256 + cc + lane_off, r);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = have ? __uint_as_float(r[x]) * p.scale : 0.f;
                    if (nc > 0) store_rows32_pairs<OUT_F32>(dk_base, wrow0, row_elems, c0 + cc, v, nc, rows_live, lane);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

struct WideDqWork {
    int b, g, hq, q0, n_kv;
    int nq, nk, off, qb, kb, vbase;  // as in BwdWork
};

// CTA index -> (b, query head, 128-row Q tile) in the dq pass's section order
// (packed batches: the order of dq_work_varlen); n_kv counts 64-key tiles, 0
// for a Q tile past the sequence's queries.
template <bool VARLEN>
__device__ __forceinline__ WideDqWork wide_dq_work(const BwdParams& p, unsigned int* err) {
    const DqWork d = VARLEN ? dq_work_varlen(p, blockIdx.x, err) : dq_work(p, blockIdx.x);
    WideDqWork w;
    w.b = d.b;
    w.g = d.g;
    w.hq = d.hq;
    w.q0 = d.q0;
    w.nq = d.nq;
    w.nk = d.nk;
    w.off = d.off;
    w.qb = d.qb;
    w.kb = d.kb;
    w.vbase = d.vbase;
    const int n_t64 = (w.nk + kWQ - 1) / kWQ;
    if (w.q0 >= w.nq) {
        w.n_kv = 0;
    } else if (p.causal) {
        const int last_row = (w.q0 + kBT - 1 < w.nq - 1 ? w.q0 + kBT - 1 : w.nq - 1);
        const int last_key = last_row + w.off;
        const int n = last_key < 0 ? 0 : last_key / kWQ + 1;
        w.n_kv = n < n_t64 ? n : n_t64;
    } else {
        w.n_kv = n_t64;
    }
    return w;
}

template <bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_wide_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                        const __grid_constant__ CUtensorMap tk64, const __grid_constant__ CUtensorMap tv64,
                        const BwdParams p, unsigned int* err) {
    using C = WideDqCfg;
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
    uint8_t* smem = reinterpret_cast<uint8_t*>((raw + 1023) & ~uintptr_t(1023));
    if ((uintptr_t)(smem - smem_raw) + C::kLayout > (uintptr_t)C::kSmemBytes) {
        if (threadIdx.x == 0) atomicOr(err, kErrLayout);
        return;
    }
    WideDqBars* bars = reinterpret_cast<WideDqBars*>(smem + C::kBar);
    const volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WideDqWork w = wide_dq_work<VARLEN>(p, err);
    auto raise_abort = [&]() {
        atomicOr(err, kErrTimeout);
        *((volatile int*)&bars->abort) = 1;
    };
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->res_full), 1);
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(smem_u32(&bars->k_full[b2]), 1);
            mbar_init(smem_u32(&bars->k_empty[b2]), 1);  // the dQ commit (S has read K before it)
            mbar_init(smem_u32(&bars->s_full[b2]), 1);
        }
        mbar_init(smem_u32(&bars->v_full), 1);
        mbar_init(smem_u32(&bars->v_empty), 1);  // the dP commit
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->ds_full), 4);
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tk64);
        tma_prefetch_desc(&tv64);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const size_t bh = (size_t)w.b * p.Hq + w.hq;
    // the K/V head and the Q / dO head as the tensor maps index them
    const int kvh = VARLEN ? w.g : w.b * p.Hkv + w.g;
    const int qh = VARLEN ? w.hq : (int)bh;

    if (warp == 0) {
        // ---- producer: Q, dO once; K_j into buffer j & 1 once dQ(j-2) has read
        // it; V_j into its one buffer once dP(j-1) has read it.
        const bool leader = elect_one();
        if (leader) {
            const uint32_t bar = smem_u32(&bars->res_full);
            mbar_arrive_expect_tx(bar, 2 * C::kBig);
#pragma unroll
            for (int c = 0; c < kWD / 64; ++c) {
                if constexpr (VARLEN) {
                    const int r = kRaggedWindow - w.nq + w.q0;
                    tma_load_5d(smem_u32(smem + C::kQ) + c * 16384, &tq, bar, 64 * c, qh, r, w.qb + w.nq,
                                kRaggedWindow);
                    tma_load_5d(smem_u32(smem + C::kDO) + c * 16384, &tdo, bar, 64 * c, qh, r, w.qb + w.nq,
                                kRaggedWindow);
                } else {
                    tma_load_3d(smem_u32(smem + C::kQ) + c * 16384, &tq, bar, 64 * c, w.q0, qh);
                    tma_load_3d(smem_u32(smem + C::kDO) + c * 16384, &tdo, bar, 64 * c, w.q0, qh);
                }
            }
        }
        __syncwarp();
        // the 64-key tile j of K or V (packed: rows past the sequence's keys
        // read as zeros)
        auto load_keys = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int j) {
#pragma unroll
            for (int c = 0; c < kWD / 64; ++c) {
                if constexpr (VARLEN)
                    tma_load_5d(dst + c * 8192, map, bar, 64 * c, kvh, kRaggedWindow - w.nk + j * kWQ,
                                w.kb + w.nk, kRaggedWindow);
                else
                    tma_load_3d(dst + c * 8192, map, bar, 64 * c, j * kWQ, kvh);
            }
        };
        bool ok = true;
        int nk = 0, nv = 0;  // K and V tiles issued
        auto load_k = [&](int j) {
            const int kb = j & 1;
            if (j >= 2)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->k_empty[kb]), ((j >> 1) - 1) & 1,
                                                       abort_flag));
            if (!ok) return;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->k_full[kb]);
                mbar_arrive_expect_tx(bar, C::kSmall);
                load_keys(smem_u32(smem + C::kK + kb * C::kSmall), &tk64, bar, j);
            }
            __syncwarp();
            ++nk;
        };
        auto load_v = [&](int j) {
            if (j >= 1)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->v_empty), (j - 1) & 1, abort_flag));
            if (!ok) return;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->v_full);
                mbar_arrive_expect_tx(bar, C::kSmall);
                load_keys(smem_u32(smem + C::kV), &tv64, bar, j);
            }
            __syncwarp();
            ++nv;
        };
        // K_0, V_0, K_1, then V_j and K_{j+1} as their buffers free up
        if (w.n_kv > 0) {
            load_k(0);
            if (ok) load_v(0);
            if (ok && w.n_kv > 1) load_k(1);
            for (int j = 1; j < w.n_kv && ok; ++j) {
                load_v(j);
                if (ok && j + 1 < w.n_kv) load_k(j + 1);
            }
        }
        if (!ok && leader) raise_abort();
        mbar_wait(smem_u32(&bars->res_full), 0, nullptr);
        for (int kb = 0; kb < 2 && kb < nk; ++kb) {
            const int uses = (nk - kb + 1) / 2;
            mbar_wait(smem_u32(&bars->k_full[kb]), (uses - 1) & 1, nullptr);
        }
        if (nv > 0) mbar_wait(smem_u32(&bars->v_full), (nv - 1) & 1, nullptr);
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer: S_0, dP_0, S_1; per tile j, once dS_j is in TMEM: dQ +=
        // dS_j K_j, dP_{j+1} (into the dP columns the dS warps have read), S_{j+2}
        // into the buffer dQ_j has read (one CTA's MMAs run in issue order).
        const bool leader = elect_one();
        const uint32_t idS = make_idesc_bf16(128, kWQ, 0, 0);
        const uint32_t idQ = make_idesc_bf16(128, kWD, 0, 1);
        const uint32_t tdP = tmem + 128, tdQ = tmem + 192;
        auto tS = [&](int j) { return tmem + (uint32_t)(j & 1) * 64u; };
        const uint32_t q_lo = sdesc_lo(smem_u32(smem + C::kQ), 16);
        const uint32_t do_lo = sdesc_lo(smem_u32(smem + C::kDO), 16);
        const uint32_t v_lo = sdesc_lo(smem_u32(smem + C::kV), 16);
        auto k_lo = [&](int kb) { return sdesc_lo(smem_u32(smem + C::kK + kb * C::kSmall), 16); };
        auto k_mn = [&](int kb) { return sdesc_lo(smem_u32(smem + C::kK + kb * C::kSmall), 8192); };
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, 32));
        };
        auto issue_s = [&](int j) {  // S_j = Q K_j^T into buffer j & 1
            if (!wait_all(smem_u32(&bars->k_full[j & 1]), (j >> 1) & 1)) return false;
            tc_fence_after();
            wbwd_issue_s(tS(j), q_lo, k_lo(j & 1), idS);
            mma_commit_warp(smem_u32(&bars->s_full[j & 1]));
            return true;
        };
        auto issue_dp = [&](int j) {  // dP_j = dO V_j^T
            if (!wait_all(smem_u32(&bars->v_full), j & 1)) return false;
            tc_fence_after();
            wbwd_issue_s(tdP, do_lo, v_lo, idS);
            mma_commit_warp(smem_u32(&bars->v_empty));  // V_j is read
            mma_commit_warp(smem_u32(&bars->dp_full));
            return true;
        };
        bool ok = true;
        if (w.n_kv > 0) {
            ok = wait_all(smem_u32(&bars->res_full), 0);
            if (ok) ok = issue_s(0);
            if (ok) ok = issue_dp(0);
            if (ok && w.n_kv > 1) ok = issue_s(1);
        }
        for (int j = 0; j < w.n_kv && ok; ++j) {
            ok = wait_all(smem_u32(&bars->ds_full), j & 1);
            if (!ok) break;
            tc_fence_after();
            wbwd_issue_ta(tdQ, tS(j), k_mn(j & 1), idQ, j > 0);    // dQ += dS_j K_j
            mma_commit_warp(smem_u32(&bars->k_empty[j & 1]));     // K_j is read (S_j, dQ_j)
            if (j + 1 < w.n_kv && !(ok = issue_dp(j + 1))) break;
            if (j + 2 < w.n_kv && !(ok = issue_s(j + 2))) break;
        }
        if (ok && w.n_kv > 0) mma_commit_warp(smem_u32(&bars->acc_full));
        if (!ok && leader) raise_abort();
        mma_commit_warp(smem_u32(&bars->drain));
        mbar_wait(smem_u32(&bars->drain), 0, nullptr);
        __syncwarp();
    } else if (warp >= 4) {
        // ---- dS (one query row per thread), then the dQ epilogue
        const int wq = warp & 3;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const uint32_t tdP = tmem + 128 + lane_off;
        const int row = w.q0 + wq * 32 + lane;
        const size_t vrow = VARLEN ? (size_t)w.hq * p.vstride + (size_t)(w.vbase + row)
                                   : bh * p.Nq_pad + row;
        // +inf past the last query: P = 0 (a tile with no work reads nothing)
        const float lse2 = w.n_kv > 0 ? p.lse2[vrow] : INFINITY;
        const float dval = w.n_kv > 0 ? p.dvec[vrow] : 0.f;
        const uint64_t c2 = f2(p.c, p.c), nl2 = f2(-lse2, -lse2), nd2 = f2(-dval, -dval);
        bool ok = true;
        for (int j = 0; j < w.n_kv && ok; ++j) {
            const uint32_t tS = tmem + (uint32_t)(j & 1) * 64u + lane_off;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->s_full[j & 1]), (j >> 1) & 1,
                                                   abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            const int lim = row + w.off - j * kWQ;  // causal: key column c allowed iff c <= lim
            const bool masked = __any_sync(0xFFFFFFFFu, p.causal && lim < kWQ - 1);
            float pf0[32], pf1[32];
            {
                uint32_t sv[32];
                tmem_ld32(tS, sv);
                tmem_wait_ld();
                if (masked) p_row_chunk<true>(sv, c2, nl2, 0, p.causal ? lim : kWQ, pf0);
                else p_row_chunk<false>(sv, c2, nl2, 0, kWQ, pf0);
                tmem_ld32(tS + 32, sv);
                tmem_wait_ld();
                if (masked) p_row_chunk<true>(sv, c2, nl2, 32, p.causal ? lim : kWQ, pf1);
                else p_row_chunk<false>(sv, c2, nl2, 32, kWQ, pf1);
            }
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->dp_full), j & 1, abort_flag, 32));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dp[32], dd[16];
                tmem_ld32(tdP, dp);
                tmem_wait_ld();
                ds_row_chunk(pf0, dp, nd2, dd);
                tmem_st16(tS, dd);
                tmem_ld32(tdP + 32, dp);
                tmem_wait_ld();
                ds_row_chunk(pf1, dp, nd2, dd);
                tmem_st16(tS + 16, dd);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->ds_full));
        }
        if (ok && w.n_kv > 0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->acc_full), 0, abort_flag));
            if (ok) tc_fence_after();
        }
        if (!ok) {
            raise_abort();
        } else {
            // every lane runs the (warp-collective) TMEM loads; rows past Nq store
            // nothing (packed batches: rows of Hq * d elements, the head's d
            // columns at hq * d)
            const size_t wrow0 = VARLEN ? (size_t)(w.qb + w.q0 + wq * 32) : bh * p.Nq + (size_t)(w.q0 + wq * 32);
            const int rows_live = w.nq - (w.q0 + wq * 32);
            const size_t row_elems = VARLEN ? (size_t)p.Hq * p.d_act : (size_t)p.d_act;
            void* dq_base = static_cast<uint8_t*>(p.dq) + (VARLEN ? (size_t)w.hq * p.d_act * (OUT_F32 ? 4 : 2) : 0);
#pragma unroll 1
            for (int cc = 0; cc < kWD; cc += 32) {
                float v[32];
                if (w.n_kv > 0) {
                    uint32_t r[32];
                    tmem_ld32(tmem + 192 + cc + lane_off, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]) * p.scale;
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] = 0.f;
                }
                const int nc = p.d_act - cc < 32 ? p.d_act - cc : 32;
                if (nc > 0) store_rows32_pairs<OUT_F32>(dq_base, wrow0, row_elems, cc, v, nc, rows_live, lane);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool OUT_F32, bool VARLEN = false>
attn_status_t launch_bwd_wide_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const CUtensorMap& tq64,
                                const CUtensorMap& tk64, const CUtensorMap& tv64,
                                const CUtensorMap& tdo64, const BwdParams& p, const void* o,
                                int o_f32, const void* dout, const float* lse, float* lse2,
                                float* dvec, cudaStream_t stream, const DeviceInfo& dev) {
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_bwd_wide_dkdv_kernel<OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WideDkdvCfg::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(attn_bwd_wide_dq_kernel<OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WideDqCfg::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    attn_status_t st;
    if constexpr (VARLEN) {
        st = launch_bwd_prep_varlen(o, o_f32, dout, lse, lse2, dvec, p, stream);
    } else {
        const long long rows_pad = (long long)p.B * p.Hq * p.Nq_pad;
        st = launch_bwd_prep(o, o_f32, dout, lse, lse2, dvec, rows_pad, p.Nq, p.Nq_pad, p.d_act, stream);
    }
    if (st != ATTN_OK) return st;
    const long long kv_ctas = 2ll * p.B * p.Hkv * p.n_kt;  // two column halves per key tile
    attn_bwd_wide_dkdv_kernel<OUT_F32, VARLEN><<<(unsigned)kv_ctas, kBwdThreads, WideDkdvCfg::kSmemBytes, stream>>>(
        tq64, tdo64, tk, tv, p, dev.err_word);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    const long long q_ctas = (long long)p.B * p.Hq * ((p.Nq + kBT - 1) / kBT);
    attn_bwd_wide_dq_kernel<OUT_F32, VARLEN><<<(unsigned)q_ctas, kBwdThreads, WideDqCfg::kSmemBytes, stream>>>(
        tq, tdo, tk64, tv64, p, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

size_t bwd_varlen_workspace_bytes(int B, int Hq, int total_q) {
    const size_t vstride = ((size_t)total_q + 132 * (size_t)B + 3) & ~(size_t)3;
    return 2 * (size_t)Hq * vstride * 4;
}

attn_status_t launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                const int* cu_q, const int* cu_k, int B, int Hq, int Hkv, int total_q,
                                int total_k, int max_q, int max_k, int d, int causal, float scale,
                                attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype,
                                void* workspace, cudaStream_t stream, const DeviceInfo& dev) {
    BwdParams p;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = max_q;
    p.Nk = max_k;
    p.Nq_pad = (max_q + kBT - 1) / kBT * kBT;
    p.group = Hq / Hkv;
    p.off = 0;  // per sequence (nk - nq)
    p.n_kt = (max_k + kBT - 1) / kBT;
    p.causal = causal;
    p.sec_groups = 1;
    p.c = scale * kBwdLog2e;
    p.scale = scale;
    p.d_act = d;
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.total_q = total_q;
    p.total_k = total_k;
    p.vstride = (int)(((size_t)total_q + 132 * (size_t)B + 3) & ~(size_t)3);
    float* lse2 = static_cast<float*>(workspace);
    float* dvec = lse2 + (size_t)Hq * p.vstride;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    if ((long long)B * Hkv * p.n_kt >= (1ll << 31) || (long long)B * Hq * (p.Nq_pad / kBT) >= (1ll << 31) ||
        (long long)Hq * p.vstride >= (1ll << 31))
        return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv, tdo;
    attn_status_t st;
    if ((st = encode_tmap_ragged(&tq, q, false, d, Hq, 64, kBT, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tk, k, false, d, Hkv, 64, kBT, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tv, v, false, d, Hkv, 64, kBT, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tdo, dout, false, d, Hq, 64, kBT, true)) != ATTN_OK) return st;
    const int o_f32 = o_dtype == ATTN_OUT_F32;
    const bool g32 = grad_dtype == ATTN_OUT_F32;
    if (d > 128) {
        // 64-row boxes for the streamed tiles of the wide passes
        if ((long long)B * Hkv * p.n_kt * 2 >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
        CUtensorMap tq64, tk64, tv64, tdo64;
        if ((st = encode_tmap_ragged(&tq64, q, false, d, Hq, 64, kWQ, true)) != ATTN_OK) return st;
        if ((st = encode_tmap_ragged(&tk64, k, false, d, Hkv, 64, kWQ, true)) != ATTN_OK) return st;
        if ((st = encode_tmap_ragged(&tv64, v, false, d, Hkv, 64, kWQ, true)) != ATTN_OK) return st;
        if ((st = encode_tmap_ragged(&tdo64, dout, false, d, Hq, 64, kWQ, true)) != ATTN_OK) return st;
        return g32 ? launch_bwd_wide_t<true, true>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, p, o, o_f32,
                                                   dout, lse, lse2, dvec, stream, dev)
                   : launch_bwd_wide_t<false, true>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, p, o, o_f32,
                                                    dout, lse, lse2, dvec, stream, dev);
    }
    // dK / dV output maps for the d = 128 kernel's staged stores: boxes of 32
    // rows x 128 bytes (64 bf16 or 32 fp32 columns)
    CUtensorMap tdk = tq, tdv = tq;
    if (pad_head_dim(d) == 128) {
        if ((st = encode_tmap_ragged(&tdk, dk, g32, d, Hkv, g32 ? 32 : 64, 32, true)) != ATTN_OK) return st;
        if ((st = encode_tmap_ragged(&tdv, dv, g32, d, Hkv, g32 ? 32 : 64, 32, true)) != ATTN_OK) return st;
        return g32 ? launch_bwd_t<128, true, true>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec,
                                                   stream, dev)
                   : launch_bwd_t<128, false, true>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec,
                                                    stream, dev);
    }
    return g32 ? launch_bwd_t<64, true, true>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec, stream,
                                              dev)
               : launch_bwd_t<64, false, true>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec, stream,
                                               dev);
}

size_t bwd_workspace_bytes(int B, int Hq, int Nq, int d) {
    (void)d;
    const size_t nq_pad = (size_t)((Nq + kBT - 1) / kBT) * kBT;
    return 2 * (size_t)B * Hq * nq_pad * 4;
}

attn_status_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                         attn_out_dtype_t o_dtype, attn_out_dtype_t grad_dtype, void* workspace,
                         cudaStream_t stream, const DeviceInfo& dev) {
    BwdParams p;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.Nq_pad = (Nq + kBT - 1) / kBT * kBT;
    p.group = Hq / Hkv;
    p.off = Nk - Nq;
    p.n_kt = (Nk + kBT - 1) / kBT;
    p.causal = causal;
    {
        // L2 budget per section: a group's Q and dO (bf16) and its K and V
        const long long per_group = 2ll * p.group * Nq * d * 2 + 2ll * Nk * d * 2;
        long long sgroups = (64ll << 20) / (per_group > 0 ? per_group : 1);
        if (sgroups < 1) sgroups = 1;
        if (sgroups > (long long)B * Hkv) sgroups = (long long)B * Hkv;
        p.sec_groups = (int)sgroups;
    }
    p.c = scale * kBwdLog2e;
    p.scale = scale;
    p.d_act = d;
    const size_t rows = (size_t)B * Hq * p.Nq_pad;
    float* lse2 = static_cast<float*>(workspace);
    float* dvec = lse2 + rows;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.cu_q = p.cu_k = nullptr;
    p.total_q = p.total_k = p.vstride = 0;
    if ((long long)B * Hkv * p.n_kt >= (1ll << 31) ||
        (long long)B * Hq * (p.Nq_pad / kBT) >= (1ll << 31))
        return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv, tdo;
    attn_status_t st;
    if ((st = encode_tmap_bf16_3d(&tq, q, d, Nq, (long long)B * Hq, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tk, k, d, Nk, (long long)B * Hkv, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tv, v, d, Nk, (long long)B * Hkv, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tdo, dout, d, Nq, (long long)B * Hq, kBT)) != ATTN_OK) return st;
    const int o_f32 = o_dtype == ATTN_OUT_F32;
    const bool g32 = grad_dtype == ATTN_OUT_F32;
    if (d > 128) {
        // 64-row boxes for the streamed tiles of the wide passes
        if ((long long)B * Hkv * p.n_kt * 2 >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
        CUtensorMap tq64, tk64, tv64, tdo64;
        if ((st = encode_tmap_bf16_3d(&tq64, q, d, Nq, (long long)B * Hq, kWQ)) != ATTN_OK) return st;
        if ((st = encode_tmap_bf16_3d(&tk64, k, d, Nk, (long long)B * Hkv, kWQ)) != ATTN_OK) return st;
        if ((st = encode_tmap_bf16_3d(&tv64, v, d, Nk, (long long)B * Hkv, kWQ)) != ATTN_OK) return st;
        if ((st = encode_tmap_bf16_3d(&tdo64, dout, d, Nq, (long long)B * Hq, kWQ)) != ATTN_OK) return st;
        return g32 ? launch_bwd_wide_t<true>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, p, o, o_f32,
                                             dout, lse, lse2, dvec, stream, dev)
                   : launch_bwd_wide_t<false>(tq, tk, tv, tdo, tq64, tk64, tv64, tdo64, p, o, o_f32,
                                              dout, lse, lse2, dvec, stream, dev);
    }
    if (pad_head_dim(d) == 128) {
        // dK / dV output maps for the staged stores: boxes of 32 rows x 128 bytes
        CUtensorMap tdk, tdv;
        if (g32) {
            if ((st = encode_tmap_f32_sw128_3d(&tdk, dk, d, Nk, (long long)B * Hkv, 32)) != ATTN_OK) return st;
            if ((st = encode_tmap_f32_sw128_3d(&tdv, dv, d, Nk, (long long)B * Hkv, 32)) != ATTN_OK) return st;
        } else {
            if ((st = encode_tmap_bf16_3d(&tdk, dk, d, Nk, (long long)B * Hkv, 32)) != ATTN_OK) return st;
            if ((st = encode_tmap_bf16_3d(&tdv, dv, d, Nk, (long long)B * Hkv, 32)) != ATTN_OK) return st;
        }
        return g32 ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec, stream,
                                             dev)
                   : launch_bwd_t<128, false>(tq, tk, tv, tdo, tdk, tdv, p, o, o_f32, dout, lse, lse2, dvec, stream,
                                              dev);
    }
    if (pad_head_dim(d) == 64)
        return g32 ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tq, tq, p, o, o_f32, dout, lse, lse2, dvec, stream, dev)
                   : launch_bwd_t<64, false>(tq, tk, tv, tdo, tq, tq, p, o, o_f32, dout, lse, lse2, dvec, stream, dev);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace gb300
