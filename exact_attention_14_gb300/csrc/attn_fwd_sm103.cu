// attn_fwd_sm103.cu -- fused exact attention forward for sm_103a.
//
// One persistent CTA per SM takes work items from the list of fwd_sched.h in
// list order: CTA i starts with item i, then fetches its next item from a
// global counter whenever it is ready for one (greedy list scheduling: with the
// causal list sorted longest-first this is LPT).  An item is a unit -- two
// 128-row Q tiles of one (batch, query head), both streaming the same K/V
// tiles -- or, for the tail units of a non-causal launch, a piece of a unit's
// KV range (fwd_sched.h, tail split).  Roles (12 warps = 3 warpgroups):
//   warp 0      TMA producer (one elected lane issues): fetches the item,
//               decodes it and hands it to the other roles through a two-slot
//               ring in shared memory, then loads the Q tiles once per item
//               and K_j, V_j into a ring of shared-memory slots (128-byte
//               swizzle, mbarrier full/empty pairs).
//   warp 1      MMA issuer (one elected lane issues): S_t = Q_t K_j^T and O_t += P_t V_j
//               on the 5th-generation tensor cores, accumulating in TMEM.
//   warps 4-7   softmax for Q tile 0, warps 8-11 for Q tile 1: one thread
//               per query row reads its S row from TMEM, applies the causal
//               / tail mask, keeps the running max m and sum l (base 2,
//               conditional rescaling with threshold tau = 8), writes P as
//               bf16 into TMEM over its S columns, and at the end of the
//               unit normalises O by 1/l and writes O and the logsumexp.
//               Two row sums are kept: lx over the unrounded P (the softmax
//               denominator the LSE needs) and l = lx plus, per tile, the
//               rounding error of the tile's largest bf16 P, which normalises
//               O (a row dominated by one key then gets exactly that V row).
//               A warp reaches TMEM lanes 32*(warp % 4) .. +31, so each
//               warpgroup covers the tile's 128 rows.
//   warps 2-3   idle.
// Registers: launched at 168 per thread; the first warpgroup (producer, MMA
// issuer) gives back to 104 and the softmax warpgroups take 200 each
// (128*104 + 256*200 = 384*168, the launch allocation; no spills).
// While one tile's softmax runs, the tensor cores work on the other tile
// (two-tile ping-pong), so exp and MMA overlap.
//
// Method: lecture notes "Optimizing Attention for Modern Hardware:
// FlashAttention 1-4" -- 2.2 online softmax and rescaling, 2.5 causal block
// skipping with an in-tile mask from global indices, 2.6 / 3.2 delayed
// normalisation and the logsumexp output, 4.5 persistent kernel, 5.3
// conditional rescaling (tau = 8 in base 2, whole-warp decision); "Flash
// Attention 3/4 notes", FA4 section 1 (two Q tiles per CTA, P through TMEM,
// 128-row tiles).
//
// TMEM columns (512 allocated): S0 [0,128) S1 [128,256) O0 [256,256+D)
// O1 [256+D, 256+2D).  P_t (bf16 pairs) overwrites S_t columns [0, 64).
#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "fwd_sched.h"

namespace gb300 {
namespace {

constexpr int kThreads = 384;
constexpr int kRegsControl = 104;  // warpgroup 0 after setmaxnreg
constexpr int kRegsSoftmax = 200;  // warpgroups 1-2 after setmaxnreg
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr float kTau = 8.0f;                    // rescale threshold (log2 units)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr uint32_t kNegInfBits = 0xFF800000u;

template <int D>
struct FwdCfg {
    static constexpr int kTileBytes = 128 * D * 2;        // one 128-row bf16 tile
    static constexpr int kStages = (D == 128) ? 4 : 8;     // K/V ring slots
    static constexpr int kRingOff = 2 * kTileBytes;        // after Q0, Q1
    // per softmax warp, two 2 KiB buffers (32 rows x 64 B) in which the merging
    // piece of a split unit stages O for TMA stores (whole units write O from
    // registers)
    static constexpr int kStgOff = kRingOff + kStages * kTileBytes;
    static constexpr int kStgBytesPerWarp = 2 * 2048;
    static constexpr int kBarOff = kStgOff + 8 * kStgBytesPerWarp;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // barriers + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // TMEM column of S_t and of O_t
    static __host__ __device__ constexpr uint32_t col_s(int t) { return uint32_t(t) * 128u; }
    static __host__ __device__ constexpr uint32_t col_o(int t) { return 256u + uint32_t(t) * D; }
};

// Output columns per staged epilogue chunk: 64 bytes per row either way.
__host__ __device__ constexpr int kEpiCols(bool f32) { return f32 ? 16 : 32; }

struct FwdParams {
    FwdShape shape;
    int group;      // Hq / Hkv
    int off;        // Nk - Nq (causal alignment)
    float c;        // scale * log2(e)
    uint32_t slot;  // work-queue slot of this launch
    int d_act;      // the tensors' head dim (<= D; the tiles' columns past it are zeros)
    FwdSplit split; // tail split (fwd_sched.h)
    float* partial; // per-piece partial results of split units (NULL if none)
    void* o;        // O: [B, Hq, Nq, d_act], or [total_q, Hq, d_act] for packed batches
    // packed variable-length batches (shape.Nq / Nk are then the maximum lengths)
    const int* cu_q;  // [B + 1] row offsets of the sequences in the packed Q / O
    const int* cu_k;  // [B + 1] row offsets in the packed K / V
    int total_q, total_k;
};

// Work queues.  Per slot: word 0 the ticket counter (the next work item),
// word 1 the number of CTAs that have exited, then one arrival counter per
// (split unit, Q tile, softmax warp) for the merge of split units.  Each
// launch uses one slot; the last CTA to exit returns the slot's words to zero,
// so the next launch (or graph replay) on the slot starts from a clean queue.
// Launches rotate through the slots, so up to kQueueSlots launches may be in
// flight at the same time on different streams.
constexpr uint32_t kQueueSlots = 256;
constexpr int kQueueWords = 2 + 8 * kMaxSplitUnits;
__device__ unsigned int g_fwd_queue[kQueueSlots][kQueueWords];

// Floats of one partial block: one softmax warp's 32 rows of one piece,
// column-major ([D + 3][32]: the normalised O columns, then m, l, lx) so that
// a warp's stores and loads of a column are 128 contiguous bytes.
template <int D>
__host__ __device__ constexpr int partial_block_floats() { return (D + 3) * 32; }

// Roles that take each work item from the producer: the MMA warp and 8
// softmax warps.
constexpr int kUnitConsumers = 9;

// A work item as the producer decodes it for the other roles, so that their
// unit boundaries carry no index arithmetic.
struct WorkItem {
    int bh;         // b * Hq + hq; -1 ends every role's loop
    int mb;         // m-block: query rows [256 mb, 256 mb + 256)
    int j0;         // first KV tile of the item
    int e[2];       // end KV tile (exclusive) of Q tile 0 and 1 (<= j0: no work)
    int part;       // piece of a split unit, -1 for a whole unit
    uint32_t cell;  // split units: 8 * (unit - n_full), the unit's first merge cell
    int q0, k0;     // packed batches: first Q / K row of the sequence
    int nq, nk;     // packed batches: the sequence's query and key counts
    int pad[2];
};

struct __align__(8) Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2];
    uint64_t unit_full[2], unit_empty[2];
    uint64_t drain;
    WorkItem item[2];
    uint32_t tmem_base;
    int abort;
};

template <int D>
struct BarsFit {
    static_assert(sizeof(Bars) <= FwdCfg<D>::kBarBytes, "barrier block");
};
template struct BarsFit<64>;
template struct BarsFit<128>;

// Consumer side of the work-item hand-off (whole warp): the k-th item this
// warp takes.  Returns false on abort.
template <bool VARLEN>
__device__ __forceinline__ bool take_item(Bars* bars, uint32_t k, WorkItem& w,
                                          const volatile int* abort_flag) {
    const uint32_t i = k & 1u;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_full[i]), (k >> 1) & 1u, abort_flag)))
        return false;
    const volatile WorkItem* src = &bars->item[i];
    w.bh = src->bh;
    w.mb = src->mb;
    w.j0 = src->j0;
    w.e[0] = src->e[0];
    w.e[1] = src->e[1];
    w.part = src->part;
    w.cell = src->cell;
    if constexpr (VARLEN) {
        w.q0 = src->q0;
        w.nq = src->nq;
        w.nk = src->nk;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&bars->unit_empty[i]));
    return true;
}

__device__ __forceinline__ void raise_abort(Bars* bars, unsigned int* err) {
    atomicOr(err, kErrTimeout);
    *((volatile int*)&bars->abort) = 1;
}

// ---------------------------------------------------------------------------
// Producer: TMA loads
// ---------------------------------------------------------------------------
// Sequence b of a packed batch: its first rows and lengths.  False (and the
// error bit, from the leader) when its offsets leave the arrays, decrease, or
// give a length above the launch's maximum, a query row without keys (nk = 0),
// or, causal, more queries than keys; such a sequence is not computed.  Every
// copy of a valid sequence stays inside [q0, q0 + nq) and [k0, k0 + nk).
__device__ __forceinline__ bool varlen_seq(const FwdParams& p, int b, bool leader, int& q0,
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
__device__ void run_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                             uint8_t* smem, Bars* bars, const FwdParams& p, unsigned int* err) {
    // Run by a whole warp so that every loop value is warp-uniform; one elected
    // lane issues the copies.
    using C = FwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xFFFFFFFFu, leader)) - 1;
    unsigned int* queue = g_fwd_queue[p.slot];
    uint32_t q_issued[2] = {0u, 0u};
    long long L = 0;  // K/V loads issued
    bool ok = true;
    bool first = true;
    for (int local = 0; ok; ++local) {
        // Take the next unit and publish it (a value >= units ends the loop
        // of every role).
        const uint32_t hs = (uint32_t)local & 1u;
        if (local >= 2)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->unit_empty[hs]),
                                                   (uint32_t)((local >> 1) - 1) & 1u, abort_flag));
        if (!ok) break;
        // A CTA's first item is its own index (no atomic on the launch's
        // critical path); later ones come from the counter, after the grid.
        // Packed batches skip the items past their sequence's last query row.
        uint32_t unit = 0;
        int part = -1, bh = -1, mb = 0, j0 = 0, j1 = 0, n0 = 0, n1 = 0;
        int q0 = 0, k0 = 0, nq = s.Nq, nk = s.Nk;
        bool done = false;
        while (true) {
            uint32_t u = blockIdx.x;
            if (!first) {
                if (leader) u = gridDim.x + atomicAdd(&queue[0], 1u);
                u = __shfl_sync(0xFFFFFFFFu, u, leader_lane);
            }
            first = false;
            done = u >= split_items(p.split);
            if (done) {
                bh = -1;  // the end marker (a skipped item may have set bh)
                break;
            }
            item_of(p.split, u, unit, part);
            unit_of(s, unit, bh, mb);
            if constexpr (VARLEN) {
                if (!varlen_seq(p, bh / s.Hq, leader, q0, nq, k0, nk, err)) continue;
                if (mb * kUnitRows >= nq) continue;
            }
            break;
        }
        if (!done) {
            n0 = tile_kv_count_len(mb, 0, nq, nk, s.causal);
            n1 = tile_kv_count_len(mb, 1, nq, nk, s.causal);
            part_range(n0 > n1 ? n0 : n1, p.split.parts, part, j0, j1);
        }
        if (leader) {
            volatile WorkItem* dst = &bars->item[hs];
            dst->bh = bh;
            dst->mb = mb;
            dst->j0 = j0;
            dst->e[0] = n0 < j1 ? n0 : j1;
            dst->e[1] = n1 < j1 ? n1 : j1;
            dst->part = part;
            dst->cell = (unit - (uint32_t)p.split.n_full) * 8u;
            dst->q0 = q0;
            dst->k0 = k0;
            dst->nq = nq;
            dst->nk = nk;
            mbar_arrive(smem_u32(&bars->unit_full[hs]));
        }
        __syncwarp();
        if (done) break;
        const int b = bh / s.Hq;
        const int hq = bh - b * s.Hq;
        const int bkv = b * s.Hkv + hq / p.group;
        for (int t = 0; t < 2 && ok; ++t) {
            if (local > 0)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->q_empty[t]), (local - 1) & 1, abort_flag));
            if (!ok) break;
            if (leader) {
                const uint32_t bar = smem_u32(&bars->q_full[t]);
                mbar_arrive_expect_tx(bar, C::kTileBytes);
                const uint32_t dst = smem_u32(smem + t * C::kTileBytes);
                const int row = mb * kUnitRows + t * kTileM;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if constexpr (VARLEN)
                        tma_load_5d(dst + c * 16384, tq, bar, 64 * c, hq, kRaggedWindow - nq + row,
                                    q0 + nq, kRaggedWindow);
                    else
                        tma_load_3d(dst + c * 16384, tq, bar, 64 * c, row, bh);
                }
            }
            __syncwarp();
            ++q_issued[t];
        }
        for (int j = j0; j < j1 && ok; ++j) {
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
                    const CUtensorMap* map = which == 0 ? tk : tv;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        if constexpr (VARLEN)
                            tma_load_5d(dst + c * 16384, map, bar, 64 * c, hq / p.group,
                                        kRaggedWindow - nk + kTileN * j, k0 + nk, kRaggedWindow);
                        else
                            tma_load_3d(dst + c * 16384, map, bar, 64 * c, kTileN * j, bkv);
                    }
                }
                __syncwarp();
                ++L;
            }
        }
    }
    if (!ok && leader) raise_abort(bars, err);
    // Without split units the queue holds only the ticket counter, which no
    // role of this CTA touches any more: count this CTA out now, off the
    // kernel's tail.  (With split units the count waits for the merges; see
    // the end of the kernel.)
    if (p.split.n_split == 0 && leader) {
        __threadfence();
        if (atomicAdd(&queue[1], 1u) == gridDim.x - 1) {
            queue[0] = 0u;
            queue[1] = 0u;
        }
    }
    // Drain: every issued copy lands before the CTA may exit.
    for (int t = 0; t < 2; ++t)
        if (q_issued[t] > 0) mbar_wait(smem_u32(&bars->q_full[t]), (q_issued[t] - 1) & 1, nullptr);
    for (int slot = 0; slot < C::kStages && slot < L; ++slot) {
        const long long n_s = (L - slot + C::kStages - 1) / C::kStages;
        mbar_wait(smem_u32(&bars->kv_full[slot]), (uint32_t)((n_s - 1) & 1), nullptr);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer (single thread)
// ---------------------------------------------------------------------------
// Descriptor low words (start address >> 4, LBO >> 4) of the K-major Q/K tiles
// and the MN-major V tile; the high word (SBO = 1024 B, version, 128-B swizzle)
// is the same constant for all three.
constexpr uint32_t kDescHi = sdesc_hi_sw128(1024);

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem, int t, uint32_t q_lo, uint32_t k_lo,
                                         uint32_t idesc) {
    using C = FwdCfg<D>;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        // +16 K-elements = +32 B inside a 128-B swizzle row; every 4 steps the
        // next 64-column chunk (16 KiB further)
        const uint32_t step = (kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4);
        mma_ss_warp(tmem + C::col_s(t), sdesc_join(q_lo + step, kDescHi),
                    sdesc_join(k_lo + step, kDescHi), idesc, kk > 0 ? 1u : 0u);
    }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem, int t, uint32_t v_lo, uint32_t idesc,
                                         bool accumulate) {
    using C = FwdCfg<D>;
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk) {
        // +16 keys = +16 rows of 128 B
        mma_ts_warp(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8,
                    sdesc_join(v_lo + kk * (2048 >> 4), kDescHi), idesc,
                    (accumulate || kk > 0) ? 1u : 0u);
    }
}

template <int D>
__device__ void run_mma(uint8_t* smem, Bars* bars, uint32_t tmem, const FwdParams& p,
                        unsigned int* err) {
    // Run by a whole warp (warp-uniform descriptors and loop state); one elected
    // lane issues every MMA and commit (elect.sync inside each instruction
    // block), so the commits track all of its MMAs.  A single issuer keeps each
    // tile's PV and S MMAs contiguous in the tensor pipe's queue.
    using C = FwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idS = make_idesc_bf16(128, kTileN, 0, 0);
    const uint32_t idO = make_idesc_bf16(128, D, 0, 1);
    // descriptor low words: Q tiles, and every ring slot as a K (LBO unused) or
    // a V (LBO = 16 KiB between the two 64-column halves) operand
    const uint32_t q_lo[2] = {sdesc_lo(smem_u32(smem), 16), sdesc_lo(smem_u32(smem + C::kTileBytes), 16)};
    const uint32_t ring = smem_u32(smem + C::kRingOff);
    auto k_lo = [&](int slot) { return sdesc_lo(ring + slot * C::kTileBytes, 16); };
    auto v_lo = [&](int slot) { return sdesc_lo(ring + slot * C::kTileBytes, 16384); };
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag));
    };
    long long Cn = 0;  // K/V loads consumed
    uint32_t cnt_p[2] = {0u, 0u};
    bool ok = true;
    for (int local = 0; ok; ++local) {
        WorkItem w;
        ok = take_item<false>(bars, (uint32_t)local, w, abort_flag);
        if (!ok || w.bh < 0) break;
        // this item's KV tiles: [j0, j1) overall, [j0, n[t]) for tile t
        const int n[2] = {w.e[0], w.e[1]};
        const int j0 = w.j0;
        const int j1 = n[0] > n[1] ? n[0] : n[1];
        // K_0 -> S_t(0).  Each tile's first S waits only for its own Q tile:
        // with causal masking the previous unit frees Q_1 only at its last
        // step, so the next unit's Q_1 lands later than its Q_0.
        int slot_k = (int)(Cn % C::kStages);
        ok = wait_all(smem_u32(&bars->kv_full[slot_k]), (uint32_t)((Cn / C::kStages) & 1));
        ++Cn;
        for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_all(smem_u32(&bars->q_full[t]), local & 1);
            if (!ok) break;
            tc_fence_after();
            if (n[t] > j0) {
                issue_qk<D>(tmem, t, q_lo[t], k_lo(slot_k), idS);
                mma_commit_warp(smem_u32(&bars->s_full[t]));
            }
            if (n[t] - j0 <= 1) mma_commit_warp(smem_u32(&bars->q_empty[t]));
        }
        if (!ok) break;
        mma_commit_warp(smem_u32(&bars->kv_empty[slot_k]));
        for (int j = j0; j < j1 && ok; ++j) {
            const int slot_v = (int)(Cn % C::kStages);
            ok = wait_all(smem_u32(&bars->kv_full[slot_v]), (uint32_t)((Cn / C::kStages) & 1));
            ++Cn;
            if (!ok) break;
            tc_fence_after();
            // K_{j+1} is awaited only when the first S(j+1) is about to be issued,
            // so a late K load never holds back the P.V of this step.
            bool k_ready = false;
            for (int t = 0; t < 2 && ok; ++t) {
                if (j >= n[t]) continue;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->p_full[t]), cnt_p[t] & 1, abort_flag, 32));
                ++cnt_p[t];
                if (!ok) break;
                tc_fence_after();
                issue_pv<D>(tmem, t, v_lo(slot_v), idO, j > j0);
                if (j + 1 < n[t]) {
                    if (!k_ready) {
                        slot_k = (int)(Cn % C::kStages);
                        ok = wait_all(smem_u32(&bars->kv_full[slot_k]), (uint32_t)((Cn / C::kStages) & 1));
                        ++Cn;
                        if (!ok) break;
                        tc_fence_after();
                        k_ready = true;
                    }
                    // Issued after PV_t(j): the tensor pipe runs this CTA's MMAs in
                    // order, so S_t(j+1) overwrites P_t(j) only once PV_t(j) has read it.
                    issue_qk<D>(tmem, t, q_lo[t], k_lo(slot_k), idS);
                    mma_commit_warp(smem_u32(&bars->s_full[t]));
                    if (j + 2 == n[t]) mma_commit_warp(smem_u32(&bars->q_empty[t]));
                } else {
                    mma_commit_warp(smem_u32(&bars->o_full[t]));
                }
            }
            if (!ok) break;
            mma_commit_warp(smem_u32(&bars->kv_empty[slot_v]));
            // k_ready holds exactly when j + 1 < j1: the producer loaded K_{j+1}
            if (k_ready) mma_commit_warp(smem_u32(&bars->kv_empty[slot_k]));
        }
    }
    if (!ok && leader) raise_abort(bars, err);
    // Drain: all issued MMAs complete before TMEM is released.
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue warpgroup (one thread per query row)
// ---------------------------------------------------------------------------
// One KV tile of the online softmax for this thread's query row: the causal /
// tail mask (MASKED only: with the mask in a separate instantiation, the
// unmasked tiles carry no per-element compare or select), the tile max, the
// conditional rescale of O (tau), P = 2^(s*c - m) rounded to bf16 into TMEM
// over the S columns, and the row sums: lx over the unrounded P (the softmax
// denominator, for the LSE) and l, which normalises O: lx plus the rounding
// error of the tile's largest P, so that the weight of the dominant key of a
// tile in O is exactly its rounded P over the sum.
template <int D, bool MASKED>
__device__ __forceinline__ void softmax_tile(uint32_t (&sr)[128], int lim, int j, float c,
                                             uint32_t tS, uint32_t tO, float& m, float& l,
                                             float& lx) {
    if constexpr (MASKED) {
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
            if (cc > lim) sr[cc] = kNegInfBits;
    }
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 128; cc += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[cc + 2]), __uint_as_float(sr[cc + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[cc + 4]), __uint_as_float(sr[cc + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[cc + 6]), __uint_as_float(sr[cc + 7]));
    }
    const float mt = fmax3(fmaxf(mx0, mx1), mx2, mx3) * c;
    const bool need = mt > m + kTau;
    if (__any_sync(0xFFFFFFFFu, need)) {
        const float m_new = fmaxf(m, mt);
        const float alpha = ex2(m - m_new);
        l *= alpha;
        lx *= alpha;
        if (j > 0) {
            // O_t is stable here: S_t(j) completing implies PV_t(j-1) completed.
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
    // rounding error of the tile's largest probability (same arithmetic as below)
    {
        const float pmax = ex2(fmaf(fmax3(fmaxf(mx0, mx1), mx2, mx3), c, -m));
        l += bf16lo_to_f32(pack_bf16x2(pmax, 0.f)) - pmax;
    }
    // p = 2^(s*c - m) on pairs; P rounded to bf16 into TMEM; unrounded row sum
    const uint64_t c2 = f2(c, c), nm2 = f2(-m, -m);
    uint64_t acc_x0 = 0, acc_x1 = 0, acc_x2 = 0, acc_x3 = 0;  // (0.f, 0.f) pairs
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int col = cc * 32 + 2 * i;
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), c2, nm2), x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if constexpr (MASKED) {
                p0 = col <= lim ? p0 : 0.f;
                p1 = col + 1 <= lim ? p1 : 0.f;
            }
            pk[i] = pack_bf16x2(p0, p1);
            switch (i & 3) {
                case 0: acc_x0 = f2_add(acc_x0, f2(p0, p1)); break;
                case 1: acc_x1 = f2_add(acc_x1, f2(p0, p1)); break;
                case 2: acc_x2 = f2_add(acc_x2, f2(p0, p1)); break;
                default: acc_x3 = f2_add(acc_x3, f2(p0, p1)); break;
            }
        }
        tmem_st16(tS + cc * 16, pk);
    }
    {
        float a, b;
        f2_split(f2_add(f2_add(acc_x0, acc_x1), f2_add(acc_x2, acc_x3)), a, b);
        lx += a + b;
        l += a + b;
    }
}

// Store of 32 output columns [cc, cc + 32) of this warp's 32 rows by the
// piece of a split unit that merges (whole units write O from registers, see
// store_o_pairs): staged 32 rows x 64 bytes at a time in shared memory (two
// buffers per warp) and written by TMA stores (rows past Nq are clipped by the
// hardware).  Packed batches are never split, so the rows are (row0, bh).
template <bool OUT_F32>
__device__ __forceinline__ void store_o_cols(const float (&v)[32], int cc, uint8_t* stg,
                                             uint32_t& epi_buf, int lane, const CUtensorMap* to,
                                             int row0, int bh, int d_act) {
    constexpr int kCols = kEpiCols(OUT_F32);
#pragma unroll
    for (int h = 0; h < 32 / kCols; ++h) {
        if (cc + h * kCols >= d_act) break;  // columns past the head dim (a box that
                                             // crosses it is clipped by the hardware)
        uint8_t* buf = stg + (epi_buf & 1) * 2048;
        if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
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

// Epilogue store of 32 output columns [cc, cc + 32) of this warp's 32 rows
// of O straight from registers, whole 32-byte sectors per store: lanes 2k and
// 2k+1 (rows 2k and 2k+1) swap one 16-byte piece of each sector, then both
// write row 2k's sector (first 16 bytes from lane 2k, second from lane 2k+1)
// and, in the next store, row 2k+1's.  No shared memory is involved (the
// tensor cores' operand reads keep it busy), and nothing waits for the
// stores to complete.
//   o_warp      address of the warp's first row of O
//   row_stride  bytes from one row of O to the next
//   rows_live   rows of the warp inside the sequence (may be <= 0)
template <bool OUT_F32>
__device__ __forceinline__ void store_o_pairs(const float (&v)[32], int cc, int lane, uint8_t* o_warp,
                                              size_t row_stride, int rows_live, int d_act) {
    constexpr int kEs = OUT_F32 ? 4 : 2;
    constexpr int kPieces = 32 * kEs / 16;  // 16-byte pieces of the row's 32 columns
    constexpr int kColsPerPiece = 16 / kEs;
    uint32_t w[kPieces * 4];
    if constexpr (OUT_F32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
    const bool odd = lane & 1;
    const int row_a = lane & ~1, row_b = lane | 1;
    uint8_t* pa = o_warp + (size_t)row_a * row_stride + (odd ? 16 : 0);
    uint8_t* pb = o_warp + (size_t)row_b * row_stride + (odd ? 16 : 0);
    const bool live_a = row_a < rows_live, live_b = row_b < rows_live;
#pragma unroll
    for (int sct = 0; sct < kPieces / 2; ++sct) {
        if (cc + 2 * sct * kColsPerPiece >= d_act) break;  // columns past the head dim
        const int pe = 2 * sct, po = 2 * sct + 1;  // the sector's two pieces
        // (d_act % 8 == 0: a piece is wholly inside or outside the row; the
        // odd lane's piece may be outside when the even lane's is not)
        const bool col_ok = cc + (odd ? po : pe) * kColsPerPiece < d_act;
        uint32_t x[4], y[4], da[4], db[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = odd ? w[pe * 4 + i] : w[po * 4 + i];  // the piece the partner writes
            y[i] = __shfl_xor_sync(0xFFFFFFFFu, x[i], 1);
            da[i] = odd ? y[i] : w[pe * 4 + i];          // row 2k: piece pe (even lane), po (odd lane)
            db[i] = odd ? w[po * 4 + i] : y[i];          // row 2k+1
        }
        const size_t off = (size_t)(cc * kEs + sct * 32);
        if (live_a && col_ok) *reinterpret_cast<uint4*>(pa + off) = make_uint4(da[0], da[1], da[2], da[3]);
        if (live_b && col_ok) *reinterpret_cast<uint4*>(pb + off) = make_uint4(db[0], db[1], db[2], db[3]);
    }
}

// End of a piece of a split unit (one softmax warp, its 32 rows of Q tile t):
// publish this warp's partial block (O / l, m, l, lx), then count the pieces
// that have arrived; the last one merges all of them (lecture notes 2.2
// rescaling, 6.1 split-KV): with M = max m_p and w_p = 2^(m_p - M),
//   O = sum_p w_p l_p (O_p / l_p) / sum_p w_p l_p,
//   LSE = ln2 * (M + log2 sum_p w_p lx_p).
// Kept out of line so that its registers do not weigh on the softmax loop.
template <int D, bool OUT_F32>
__device__ __noinline__ void split_piece_epilogue(unsigned int* merge_count, float* partial,
                                                  int parts, uint32_t cell, int part, int lane,
                                                  uint32_t tO, float m, float l, float lx,
                                                  uint8_t* stg, uint32_t* epi_buf,
                                                  const CUtensorMap* to, int row0, int bh,
                                                  float* lse_out, int d_act) {
    const float inv_l = 1.0f / l;
    float* blocks = partial + (size_t)cell * parts * partial_block_floats<D>();
    float* mine = blocks + (size_t)part * partial_block_floats<D>();
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
        uint32_t r[32];
        tmem_ld32(tO + cc, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) mine[(cc + i) * 32 + lane] = __fmul_rn(__uint_as_float(r[i]), inv_l);
    }
    mine[D * 32 + lane] = m;
    mine[(D + 1) * 32 + lane] = l;
    mine[(D + 2) * 32 + lane] = lx;
    __threadfence();
    __syncwarp();
    uint32_t arrived = 0;
    if (lane == 0) arrived = atomicAdd(&merge_count[cell], 1u);
    arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
    if (arrived != (uint32_t)parts - 1) return;
    // The last piece merges, summing the pieces in piece order with the
    // same arithmetic whichever piece arrives last (so the result does not
    // depend on the arrival order).  Its own O / l is recomputed from TMEM
    // exactly as it was written; the other pieces' blocks come from L2,
    // the first other piece's next 32-column chunk loaded ahead of use.
    __threadfence();
    float mq[kMaxSplitParts], lq[kMaxSplitParts], lxq[kMaxSplitParts];
#pragma unroll
    for (int q = 0; q < kMaxSplitParts; ++q) {
        mq[q] = -INFINITY; lq[q] = 0.f; lxq[q] = 0.f;
        if (q == part) {
            mq[q] = m; lq[q] = l; lxq[q] = lx;
        } else if (q < parts) {
            const float* bq = blocks + q * partial_block_floats<D>() + D * 32 + lane;
            mq[q] = __ldcg(bq);
            lq[q] = __ldcg(bq + 32);
            lxq[q] = __ldcg(bq + 64);
        }
    }
    float mmax = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxSplitParts; ++q) mmax = fmaxf(mmax, mq[q]);
    float wsum = 0.f, wxsum = 0.f;
    float w[kMaxSplitParts];
#pragma unroll
    for (int q = 0; q < kMaxSplitParts; ++q) {
        const float e = ex2(mq[q] - mmax);  // 0 for absent pieces
        w[q] = e * lq[q];
        wsum += w[q];
        wxsum += e * lxq[q];
    }
    const float inv_w = 1.0f / wsum;
#pragma unroll
    for (int q = 0; q < kMaxSplitParts; ++q) w[q] *= inv_w;  // weight of piece q's O / l
    const int q0 = part == 0 ? 1 : 0;
    const float* b0 = blocks + q0 * partial_block_floats<D>() + lane;
    float nxt[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) nxt[i] = __ldcg(b0 + i * 32);
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
        uint32_t r[32];
        tmem_ld32(tO + cc, r);
        float cur[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) cur[i] = nxt[i];
        if (cc + 32 < D) {
#pragma unroll
            for (int i = 0; i < 32; ++i) nxt[i] = __ldcg(b0 + (cc + 32 + i) * 32);
        }
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll 1
        for (int q = 0; q < parts; ++q) {
            float wq_ = 0.f;
#pragma unroll
            for (int x = 0; x < kMaxSplitParts; ++x) wq_ = x == q ? w[x] : wq_;
            if (q == part) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaf(wq_, __fmul_rn(__uint_as_float(r[i]), inv_l), v[i]);
            } else if (q == q0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaf(wq_, cur[i], v[i]);
            } else {
                const float* bq = blocks + q * partial_block_floats<D>() + cc * 32 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaf(wq_, __ldcg(bq + i * 32), v[i]);
            }
        }
        store_o_cols<OUT_F32>(v, cc, stg, *epi_buf, lane, to, row0, bh, d_act);
    }
    if (lse_out) *lse_out = (mmax + log2f(wxsum)) * kLn2;
}

template <int D, bool OUT_F32, bool VARLEN>
__device__ void run_softmax(int t, int wq, int lane, uint8_t* smem, Bars* bars, uint32_t tmem,
                            const FwdParams& p, const CUtensorMap* to, float* __restrict__ lse_ptr,
                            unsigned int* err) {
    using C = FwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const FwdShape& s = p.shape;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + C::col_s(t) + lane_off;
    const uint32_t tO = tmem + C::col_o(t) + lane_off;
    const uint32_t bar_s = smem_u32(&bars->s_full[t]);
    const uint32_t bar_p = smem_u32(&bars->p_full[t]);
    const uint32_t bar_o = smem_u32(&bars->o_full[t]);
    const float c = p.c;
    uint8_t* stg = smem + C::kStgOff + (t * 4 + wq) * C::kStgBytesPerWarp;
    uint32_t epi_buf = 0;
    uint32_t cnt_s = 0, cnt_o = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
        WorkItem w;
        ok = take_item<VARLEN>(bars, k, w, abort_flag);
        if (!ok || w.bh < 0) break;
        const int bh = w.bh, mb = w.mb, j0 = w.j0, part = w.part;
        const int n_t = t == 0 ? w.e[0] : w.e[1];
        if (n_t <= j0) continue;
        const int nq = VARLEN ? w.nq : s.Nq;
        const int nk = VARLEN ? w.nk : s.Nk;
        const int row = mb * kUnitRows + t * kTileM + wq * 32 + lane;
        // last allowed key for this row (index within the sequence)
        int last_key = nk - 1;
        if (s.causal) {
            const int lk = row + (VARLEN ? nk - nq : p.off);
            last_key = lk < last_key ? lk : last_key;
        }
        float m = -INFINITY;  // running max of scaled scores, log2 units
        float l = 0.f;        // normaliser of O (see softmax_tile)
        float lx = 0.f;       // running sum of the unrounded probabilities (gives the LSE)
        for (int j = j0; j < n_t; ++j) {
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
            const int lim = last_key - j * kTileN;  // column c allowed iff c <= lim
            if (__any_sync(0xFFFFFFFFu, lim < kTileN - 1))
                softmax_tile<D, true>(sr, lim, j - j0, c, tS, tO, m, l, lx);
            else
                softmax_tile<D, false>(sr, lim, j - j0, c, tS, tO, m, l, lx);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p);
        }
        if (!ok) break;
        // Epilogue: O = O_acc / l, LSE = ln2 * (m + log2 lx)
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o, cnt_o & 1, abort_flag));
        ++cnt_o;
        if (!ok) break;
        tc_fence_after();
        const bool live = row < nq;
        const float inv_l = 1.0f / l;
        const int hq = bh - (bh / s.Hq) * s.Hq;
        // LSE: [B, Hq, Nq], or [Hq, total_q] for packed batches
        const size_t row_idx = VARLEN ? (size_t)hq * p.total_q + (size_t)(w.q0 + row)
                                      : (size_t)bh * s.Nq + (size_t)row;
        const uint64_t il2 = f2(inv_l, inv_l);
        if (part < 0) {
            // this warp's first row of O and the stride between rows
            constexpr int kEs = OUT_F32 ? 4 : 2;
            const int wrow = mb * kUnitRows + t * kTileM + wq * 32;
            const size_t first = VARLEN ? (size_t)(w.q0 + wrow) * s.Hq + (size_t)hq
                                        : (size_t)bh * s.Nq + (size_t)wrow;
            uint8_t* o_warp = static_cast<uint8_t*>(p.o) + first * (size_t)p.d_act * kEs;
            const size_t row_stride = (VARLEN ? (size_t)s.Hq : 1u) * (size_t)p.d_act * kEs;
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t r[32];
                tmem_ld32(tO + cc, r);
                tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    f2_split(f2_mul(f2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), il2), v[i], v[i + 1]);
                store_o_pairs<OUT_F32>(v, cc, lane, o_warp, row_stride, nq - wrow, p.d_act);
            }
            if (live && lse_ptr) lse_ptr[row_idx] = (m + log2f(lx)) * kLn2;
            continue;
        }
        if constexpr (!VARLEN) {  // packed batches are never split
            // (cell: this warp's slot among the split units' merge counters and blocks)
            const uint32_t cell = w.cell + (uint32_t)t * 4u + (uint32_t)wq;
            const int row0 = mb * kUnitRows + t * kTileM + wq * 32;
            split_piece_epilogue<D, OUT_F32>(g_fwd_queue[p.slot] + 2, p.partial, p.split.parts, cell,
                                             part, lane, tO, m, l, lx, stg, &epi_buf, to, row0, bh,
                                             (live && lse_ptr) ? lse_ptr + row_idx : nullptr, p.d_act);
        }
    }
    if (lane == 0) bulk_wait_group_all();  // every staged store has completed
    __syncwarp();
    if (!ok) raise_abort(bars, err);
}

template <int D, bool OUT_F32, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                float* __restrict__ lse_ptr, const FwdParams p, unsigned int* err) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
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
            mbar_init(smem_u32(&bars->unit_empty[i]), kUnitConsumers);
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
        if (warp == 0) run_producer<D, VARLEN>(&tq, &tk, &tv, smem, bars, p, err);
        if (warp == 1) run_mma<D>(smem, bars, tmem, p, err);
    } else {
        reg_alloc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        run_softmax<D, OUT_F32, VARLEN>(t, warp & 3, lane, smem, bars, tmem, p, &to, lse_ptr, err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // With split units, the last CTA to exit returns the queue slot to zero:
    // the ticket counter, the exit count and the merge counters.  Every ticket
    // and merge-counter atomic of this CTA returned its value before the
    // barrier above, so they precede the exit count.
    if (p.split.n_split > 0 && threadIdx.x == 0) {
        unsigned int* queue = g_fwd_queue[p.slot];
        __threadfence();
        if (atomicAdd(&queue[1], 1u) == gridDim.x - 1) {
            __threadfence();
            const int words = 8 * p.split.n_split;
            for (int i = 0; i < words; ++i) queue[2 + i] = 0u;
            queue[0] = 0u;
            queue[1] = 0u;
        }
    }
}

template <int D, bool OUT_F32, bool VARLEN = false>
attn_status_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, float* lse, const FwdParams& p, int grid,
                           cudaStream_t stream, const DeviceInfo& dev) {
    using C = FwdCfg<D>;
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_fwd_kernel<D, OUT_F32, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    attn_fwd_kernel<D, OUT_F32, VARLEN><<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, to, lse, p, dev.err_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, bool OUT_F32>
attn_status_t launch_with_partials(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& to, float* lse,
                                   FwdParams& p, int grid, void* workspace, cudaStream_t stream,
                                   const DeviceInfo& dev) {
    // the split units' partial results live in the caller's workspace
    // (fwd_workspace_bytes of it, checked by the caller of launch_fwd)
    p.partial = p.split.n_split > 0 ? static_cast<float*>(workspace) : nullptr;
    return launch_fwd_t<D, OUT_F32>(tq, tk, tv, to, lse, p, grid, stream, dev);
}

uint32_t next_queue_slot() {
    static std::atomic<uint32_t> launches{0};
    return launches.fetch_add(1u, std::memory_order_relaxed) % kQueueSlots;
}

}  // namespace

size_t fwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int num_sms) {
    if (d > 128) return 0;  // the d > 128 kernel splits no unit
    const FwdShape s = make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal);
    const FwdSplit sp = plan_tail_split(s, num_sms);
    const size_t block = pad_head_dim(d) == 128 ? partial_block_floats<128>() : partial_block_floats<64>();
    return (size_t)sp.n_split * sp.parts * 8 * block * sizeof(float);
}

attn_status_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                         attn_out_dtype_t o_dtype, void* workspace, cudaStream_t stream,
                         const DeviceInfo& dev) {
    if (d > 128)
        return launch_fwd_wide(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, o_dtype, stream,
                               dev);
    FwdParams p;
    p.shape = make_fwd_shape(B, Hq, Hkv, Nq, Nk, d, causal, dev.num_sms);
    if (p.shape.units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    p.group = Hq / Hkv;
    p.off = Nk - Nq;
    p.c = scale * kLog2e;
    p.d_act = d;
    p.slot = next_queue_slot();
    p.split = plan_tail_split(p.shape, dev.num_sms);
    p.cu_q = p.cu_k = nullptr;
    p.total_q = p.total_k = 0;
    const uint32_t items = split_items(p.split);
    const int grid = (int)(items < (uint32_t)dev.num_sms ? items : (uint32_t)dev.num_sms);
    p.partial = nullptr;
    p.o = o;
    CUtensorMap tq, tk, tv, to;
    attn_status_t st;
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if ((st = encode_tmap_bf16_3d(&tq, q, d, Nq, (long long)B * Hq, kTileM)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tk, k, d, Nk, (long long)B * Hkv, kTileN)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tv, v, d, Nk, (long long)B * Hkv, kTileN)) != ATTN_OK) return st;
    if ((st = encode_tmap_out_3d(&to, o, f32, d, Nq, (long long)B * Hq, kEpiCols(f32), 32)) != ATTN_OK)
        return st;
    // head dims below 64 / 128 run on those kernels (TMA zero-fills the rest)
    if (pad_head_dim(d) == 128)
        return f32 ? launch_with_partials<128, true>(tq, tk, tv, to, lse, p, grid, workspace, stream, dev)
                   : launch_with_partials<128, false>(tq, tk, tv, to, lse, p, grid, workspace, stream, dev);
    if (pad_head_dim(d) == 64)
        return f32 ? launch_with_partials<64, true>(tq, tk, tv, to, lse, p, grid, workspace, stream, dev)
                   : launch_with_partials<64, false>(tq, tk, tv, to, lse, p, grid, workspace, stream, dev);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace gb300

namespace gb300 {

attn_status_t launch_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                const int* cu_q, const int* cu_k, int B, int Hq, int Hkv,
                                int total_q, int total_k, int max_q, int max_k, int d, int causal,
                                float scale, attn_out_dtype_t o_dtype, cudaStream_t stream,
                                const DeviceInfo& dev) {
    FwdParams p;
    // units cover every sequence at the maximum lengths; the producer skips
    // the m-blocks past each sequence's own length
    p.shape = make_fwd_shape(B, Hq, Hkv, max_q, max_k, d, causal);
    if (p.shape.units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    p.group = Hq / Hkv;
    p.off = 0;
    p.c = scale * kLog2e;
    p.d_act = d;
    p.slot = next_queue_slot();
    p.split.n_full = (int)p.shape.units;  // sequences differ in cost: no tail split
    p.split.n_split = 0;
    p.split.parts = 1;
    p.partial = nullptr;
    p.o = o;
    p.cu_q = cu_q;
    p.cu_k = cu_k;
    p.total_q = total_q;
    p.total_k = total_k;
    const long long items = p.shape.units;
    const int grid = (int)(items < dev.num_sms ? items : dev.num_sms);
    CUtensorMap tq, tk, tv, to;
    attn_status_t st;
    const bool f32 = o_dtype == ATTN_OUT_F32;
    if ((st = encode_tmap_ragged(&tq, q, false, d, Hq, 64, kTileM, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tk, k, false, d, Hkv, 64, kTileN, true)) != ATTN_OK) return st;
    if ((st = encode_tmap_ragged(&tv, v, false, d, Hkv, 64, kTileN, true)) != ATTN_OK) return st;
    // (O of a packed batch is written from registers, never by this map; it
    // is still encoded, which checks O's alignment like the other maps)
    if ((st = encode_tmap_ragged(&to, o, f32, d, Hq, kEpiCols(f32), 32, false)) != ATTN_OK) return st;
    if (pad_head_dim(d) == 128)
        return f32 ? launch_fwd_t<128, true, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
                   : launch_fwd_t<128, false, true>(tq, tk, tv, to, lse, p, grid, stream, dev);
    if (pad_head_dim(d) == 64)
        return f32 ? launch_fwd_t<64, true, true>(tq, tk, tv, to, lse, p, grid, stream, dev)
                   : launch_fwd_t<64, false, true>(tq, tk, tv, to, lse, p, grid, stream, dev);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace gb300
