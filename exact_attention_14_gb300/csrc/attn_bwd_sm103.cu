// attn_bwd_sm103.cu -- attention backward (dQ, dK, dV) for sm_103a.
//
// Method: lecture notes "Optimizing Attention for Modern Hardware:
// FlashAttention 1-4", 2.6 (P recomputed from the stored logsumexp,
// D = rowsum(dO o O), the K/V-outer loop with dK and dV accumulated on chip and
// dQ accumulated with atomic adds) and exercise 6; "Flash Attention 3/4
// notes", FA4 section 2 (five MMAs per tile -- S, dP, dV, dK, dQ -- with the
// accumulators in tensor memory).
//
// Three kernels:
//  prep  per query row: D = sum_c dO_c O_c and lse2 = LSE log2(e), padded to
//        whole 128-row tiles (lse2 = +inf and D = 0 past Nq, so padded rows
//        get P = 0 and dS = 0); zeroes the row of the fp32 dQ accumulator.
//  main  one CTA per (b, KV head g, 128-key tile).  K and V of the tile stay
//        in shared memory; the CTA walks every query head of g's group and
//        every 128-row Q tile that can see its keys.  Per Q tile:
//          S^T  = K Q^T,  dP^T = V dO^T      (tcgen05, operands K-major in smem)
//          P^T  = 2^(S^T c - lse2),  dS^T = P^T o (dP^T - D)
//                 (warps 4-7, one key row per thread; P^T and dS^T go to TMEM
//                 as bf16 pairs, dS^T also to shared memory as dQ's A operand)
//          dV  += P^T dO,  dK += dS^T Q      (A from TMEM, B MN-major in smem)
//          dQ   = dS K                       (A = dS MN-major, B = K MN-major)
//                 (warps 8-11 load dQ from TMEM into registers, release it,
//                 and add it into the fp32 accumulator with 16-byte atomics)
//        After the last tile dK (times scale) and dV are written once.
//  post  dQ = scale * accumulator, as bf16 or fp32.
//
// Roles of the main kernel (12 warps): warp 0 TMA producer (K, V once; Q, dO,
// lse2 and D per tile into a two-stage ring), warp 1 MMA issuer and TMEM owner,
// warps 2-3 idle, warps 4-7 P / dS, warps 8-11 dQ read-out.
//
// TMEM (512 columns): [0,128) S^T, then P^T in [0,64), then dQ in [0,d);
// [128,256) dP^T, then dS^T in [128,192); dV [256,256+d); dK [256+d,256+2d).
// S^T of the next tile is issued only once dQ of this one has been read out;
// dP^T of the next tile goes ahead of that wait (its columns are free as soon
// as dK has read dS^T, and one CTA's MMAs run in issue order).
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kBwdThreads = 384;
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
    static constexpr int kDS = 6 * kTile;       // dS^T, 128 x 128 bf16, MN-major SW128
    static constexpr int kLD = kDS + kBT * kBT * 2;  // 2 stages x (lse2[128], D[128])
    static constexpr int kBar = kLD + 2 * 1024;
    static constexpr int kLayout = kBar + 256;
    static constexpr int kSmemBytes =
        kLayout + 1024 < kMaxSmemPerBlock ? kLayout + 1024 : kMaxSmemPerBlock;
    static_assert(kLayout <= kMaxSmemPerBlock, "shared memory budget");
};

struct BwdParams {
    int B, Hq, Hkv, Nq, Nk, Nq_pad, group, off, n_kt, causal;
    int sec_groups;     // (b, KV head) groups per L2 section
    float c;      // scale * log2(e)
    float scale;
    const float* lse2;  // [B*Hq, Nq_pad]
    const float* dvec;  // [B*Hq, Nq_pad]
    float* dq_acc;      // [B*Hq, Nq_pad, d]
    void* dk;           // [B, Hkv, Nk, d]
    void* dv;
};

struct __align__(8) BwdBars {
    uint64_t kv_full;
    uint64_t qd_full[2], qd_empty[2];
    uint64_t s_full, p_full, dq_full, dq_empty, acc_full, drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

// The CTA's work: K/V tile kt of (b, g) and the Q tiles [qt_first, n_qt) of
// each query head of the group, head-major.
//
// Order of the CTAs: the (b, KV head) groups are cut into L2 sections whose
// dQ accumulator, Q, dO, K and V fit an L2 budget (so the dQ atomic adds of
// all the section's key tiles meet in L2 instead of DRAM, and each Q / dO
// tile is read from DRAM once for all of them); sections run in order, and
// inside a section key tiles are outer (causal tile 0, which sees the most
// query tiles, first).
struct BwdWork {
    int b, g, kt, k0, qt_first, n_qt_cta, n_tiles;
};

__device__ __forceinline__ BwdWork bwd_work(const BwdParams& p) {
    BwdWork w;
    const unsigned all = (unsigned)(p.B * p.Hkv);
    const unsigned S = (unsigned)p.sec_groups;
    const unsigned per_sec = S * (unsigned)p.n_kt;
    const unsigned sec = blockIdx.x / per_sec;
    const unsigned r = blockIdx.x - sec * per_sec;
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
    return w;
}

__device__ __forceinline__ void bwd_abort(BwdBars* bars, unsigned int* err) {
    atomicOr(err, kErrTimeout);
    *((volatile int*)&bars->abort) = 1;
}

// ---------------------------------------------------------------------------
// Producer
// ---------------------------------------------------------------------------
template <int D>
__device__ void bwd_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                             const CUtensorMap* tdo, uint8_t* smem, BwdBars* bars,
                             const BwdParams& p, const BwdWork& w, unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const int kvh = w.b * p.Hkv + w.g;
    if (leader) {
        const uint32_t bar = smem_u32(&bars->kv_full);
        mbar_arrive_expect_tx(bar, 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(smem_u32(smem + C::kK) + c * 16384, tk, bar, 64 * c, w.k0, kvh);
            tma_load_3d(smem_u32(smem + C::kV) + c * 16384, tv, bar, 64 * c, w.k0, kvh);
        }
    }
    __syncwarp();
    bool ok = true;
    int issued = 0;
    for (int i = 0; i < w.n_tiles && ok; ++i) {
        const int st = i & 1;
        if (i >= 2)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->qd_empty[st]), ((i >> 1) - 1) & 1,
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
                tma_load_3d(smem_u32(smem + C::kQ + st * C::kTile) + c * 16384, tq, bar, 64 * c, q0, bh);
                tma_load_3d(smem_u32(smem + C::kDO + st * C::kTile) + c * 16384, tdo, bar, 64 * c, q0, bh);
            }
            const size_t row = (size_t)bh * p.Nq_pad + q0;
            bulk_load(smem_u32(smem + C::kLD + st * 1024), p.lse2 + row, 512, bar);
            bulk_load(smem_u32(smem + C::kLD + st * 1024 + 512), p.dvec + row, 512, bar);
        }
        __syncwarp();
        ++issued;
    }
    if (!ok && leader) bwd_abort(bars, err);
    // Drain: every issued copy lands before the CTA may exit.
    mbar_wait(smem_u32(&bars->kv_full), 0, nullptr);
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

// M=128 x N=d x K=128 with A from TMEM (bf16 pairs, 8 columns per K=16) and B
// MN-major in smem (16 rows of 128 B per K=16): dV += P^T dO or dK += dS^T Q.
__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kBT / 16; ++kk)
        mma_ts_warp(d_tmem, a_tmem + kk * 8, sdesc_join(b_lo + kk * (2048 >> 4), kBwdDescHi), idesc,
                    (accumulate || kk > 0) ? 1u : 0u);
}

template <int D>
__device__ void bwd_mma(uint8_t* smem, BwdBars* bars, uint32_t tmem, const BwdWork& w,
                        unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const bool leader = elect_one();
    const uint32_t idS = make_idesc_bf16(128, 128, 0, 0);
    const uint32_t idKV = make_idesc_bf16(128, D, 0, 1);
    const uint32_t idQ = make_idesc_bf16(128, D, 1, 1);
    const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
    const uint32_t k_kmaj = sdesc_lo(smem_u32(smem + C::kK), 16);
    const uint32_t v_kmaj = sdesc_lo(smem_u32(smem + C::kV), 16);
    const uint32_t k_mn = sdesc_lo(smem_u32(smem + C::kK), 16384);
    const uint32_t ds_mn = sdesc_lo(smem_u32(smem + C::kDS), 16384);
    auto q_kmaj = [&](int st) { return sdesc_lo(smem_u32(smem + C::kQ + st * C::kTile), 16); };
    auto do_kmaj = [&](int st) { return sdesc_lo(smem_u32(smem + C::kDO + st * C::kTile), 16); };
    auto q_mn = [&](int st) { return sdesc_lo(smem_u32(smem + C::kQ + st * C::kTile), 16384); };
    auto do_mn = [&](int st) { return sdesc_lo(smem_u32(smem + C::kDO + st * C::kTile), 16384); };
    auto wait_all = [&](uint32_t bar, uint32_t parity, int polls) {
        return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, polls));
    };
    bool ok = true;
    if (w.n_tiles > 0) {
        ok = wait_all(smem_u32(&bars->kv_full), 0, 0) && wait_all(smem_u32(&bars->qd_full[0]), 0, 0);
        if (ok) {
            tc_fence_after();
            issue_kmajor<D>(tS, k_kmaj, q_kmaj(0), idS);
            issue_kmajor<D>(tdP, v_kmaj, do_kmaj(0), idS);
            mma_commit_warp(smem_u32(&bars->s_full));
        }
        for (int i = 0; i < w.n_tiles && ok; ++i) {
            const int st = i & 1;
            ok = wait_all(smem_u32(&bars->p_full), i & 1, 32);
            if (!ok) break;
            tc_fence_after();
            issue_tmem_a(tdV, tS, do_mn(st), idKV, i > 0);
            issue_tmem_a(tdK, tdP, q_mn(st), idKV, i > 0);
            mma_commit_warp(smem_u32(&bars->qd_empty[st]));  // Q and dO of this tile are read
#pragma unroll
            for (int kk = 0; kk < kBT / 16; ++kk)
                mma_ss_warp(tS, sdesc_join(ds_mn + kk * (2048 >> 4), kBwdDescHi),
                            sdesc_join(k_mn + kk * (2048 >> 4), kBwdDescHi), idQ, kk > 0 ? 1u : 0u);
            mma_commit_warp(smem_u32(&bars->dq_full));
            if (i + 1 < w.n_tiles) {
                const int st1 = (i + 1) & 1;
                ok = wait_all(smem_u32(&bars->qd_full[st1]), ((i + 1) >> 1) & 1, 0);
                if (!ok) break;
                tc_fence_after();
                issue_kmajor<D>(tdP, v_kmaj, do_kmaj(st1), idS);
                ok = wait_all(smem_u32(&bars->dq_empty), i & 1, 32);
                if (!ok) break;
                tc_fence_after();
                issue_kmajor<D>(tS, k_kmaj, q_kmaj(st1), idS);
                mma_commit_warp(smem_u32(&bars->s_full));
            }
        }
        if (ok) mma_commit_warp(smem_u32(&bars->acc_full));
    }
    if (!ok && leader) bwd_abort(bars, err);
    // Drain: all issued MMAs complete before TMEM is released.
    mma_commit_warp(smem_u32(&bars->drain));
    mbar_wait(smem_u32(&bars->drain), 0, nullptr);
    __syncwarp();
}

// ---------------------------------------------------------------------------
// P / dS warpgroup (one key row per thread) and the dK / dV epilogue
// ---------------------------------------------------------------------------
template <bool MASKED>
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                           uint32_t lse2s, uint32_t ds_vec, int qc, float c,
                                           int lim, uint32_t (&pp)[16], uint32_t (&dd)[16]) {
    // lim: query column qc + x is allowed iff qc + x >= lim (causal), else all.
    // The tile's lse2 and D come from shared memory 4 at a time (broadcast).
    const uint64_t c2 = f2(c, c);
#pragma unroll
    for (int x4 = 0; x4 < 8; ++x4) {
        const float4 l4 = lds128_f32(lse2s + 4u * (qc + 4 * x4));
        const float4 d4 = lds128_f32(ds_vec + 4u * (qc + 4 * x4));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int x = 2 * x4 + h;
            const int q = qc + 2 * x;
            const uint64_t nl = h == 0 ? f2(-l4.x, -l4.y) : f2(-l4.z, -l4.w);
            const uint64_t nd = h == 0 ? f2(-d4.x, -d4.y) : f2(-d4.z, -d4.w);
            float a0, a1;
            f2_split(f2_fma(f2(__uint_as_float(s[2 * x]), __uint_as_float(s[2 * x + 1])), c2, nl), a0, a1);
            float p0 = ex2(a0), p1 = ex2(a1);
            if constexpr (MASKED) {
                p0 = q >= lim ? p0 : 0.f;
                p1 = q + 1 >= lim ? p1 : 0.f;
            }
            float d0, d1;
            f2_split(f2_mul(f2(p0, p1), f2_add(f2(__uint_as_float(dp[2 * x]), __uint_as_float(dp[2 * x + 1])), nd)),
                     d0, d1);
            pp[x] = pack_bf16x2(p0, p1);
            dd[x] = pack_bf16x2(d0, d1);
        }
    }
}

template <int D, bool OUT_F32>
__device__ __forceinline__ void store_row32(void* base, size_t elem, const float (&v)[32]) {
    if constexpr (OUT_F32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(base) + elem);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            dst[i] = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    }
}

template <int D, bool OUT_F32>
__device__ void bwd_pds(int wq, int lane, uint8_t* smem, BwdBars* bars, uint32_t tmem,
                        const BwdParams& p, const BwdWork& w, unsigned int* err) {
    using C = BwdCfg<D>;
    const volatile int* abort_flag = &bars->abort;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off, tdP = tmem + 128 + lane_off;
    const int j = wq * 32 + lane;  // key row of the tile
    const int jg = w.k0 + j;
    const uint32_t ds_row = smem_u32(smem + C::kDS) + j * 128;
    bool ok = true;
    for (int i = 0; i < w.n_tiles && ok; ++i) {
        const int st = i & 1;
        ok = mbar_wait(smem_u32(&bars->s_full), i & 1, abort_flag, 32);
        if (!ok) break;
        tc_fence_after();
        const int q0 = (w.qt_first + i % w.n_qt_cta) * kBT;
        const uint32_t lse2s = smem_u32(smem + C::kLD + st * 1024);
        const uint32_t ds_vec = lse2s + kBT * 4;
        // causal: query q0 + x sees key jg iff x >= jg - off - q0
        const int lim = jg - p.off - q0;
        const bool masked = p.causal && (q0 + p.off < w.k0 + kBT - 1);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t s[32], dp[32];
            tmem_ld32(tS + cc * 32, s);
            tmem_ld32(tdP + cc * 32, dp);
            tmem_wait_ld();
            uint32_t pp[16], dd[16];
            if (masked)
                p_ds_chunk<true>(s, dp, lse2s, ds_vec, cc * 32, p.c, lim, pp, dd);
            else
                p_ds_chunk<false>(s, dp, lse2s, ds_vec, cc * 32, p.c, lim, pp, dd);
            tmem_st16(tS + cc * 16, pp);   // P^T over S^T columns already read
            tmem_st16(tdP + cc * 16, dd);  // dS^T over dP^T columns already read
            // dS^T row j, queries [32 cc, 32 cc + 32): four 16-byte granules of the
            // MN-major 128-byte-swizzled A operand of dQ (64-query chunks 16 KiB apart)
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                const int G = cc * 4 + gq;
                const int off = (G >> 3) * 16384 + ((((G & 7) ^ (j & 7))) << 4);
                sts128(ds_row + off, dd[4 * gq], dd[4 * gq + 1], dd[4 * gq + 2], dd[4 * gq + 3]);
            }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(smem_u32(&bars->p_full));
            mbar_arrive(smem_u32(&bars->qd_empty[st]));
        }
    }
    if (!ok) {
        bwd_abort(bars, err);
        return;
    }
    // dK = scale * dS^T Q, dV = P^T dO: one key row per thread, written once
    const bool live = jg < p.Nk;
    const size_t elem = (((size_t)w.b * p.Hkv + w.g) * p.Nk + (size_t)(live ? jg : 0)) * D;
    if (w.n_tiles == 0) {
        float z[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) z[x] = 0.f;
        if (live)
#pragma unroll 1
            for (int cc = 0; cc < D; cc += 32) {
                store_row32<D, OUT_F32>(p.dk, elem + cc, z);
                store_row32<D, OUT_F32>(p.dv, elem + cc, z);
            }
        return;
    }
    ok = mbar_wait(smem_u32(&bars->acc_full), 0, abort_flag);
    if (!ok) {
        bwd_abort(bars, err);
        return;
    }
    tc_fence_after();
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
        uint32_t r[32];
        float v[32];
        tmem_ld32(tmem + 256 + cc + lane_off, r);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]);
        if (live) store_row32<D, OUT_F32>(p.dv, elem + cc, v);
        tmem_ld32(tmem + 256 + D + cc + lane_off, r);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = __uint_as_float(r[x]) * p.scale;
        if (live) store_row32<D, OUT_F32>(p.dk, elem + cc, v);
    }
}

// ---------------------------------------------------------------------------
// dQ read-out (one query row per thread): TMEM -> fp32 accumulator.  The
// whole row is loaded into registers first and TMEM released at once (the next
// tile's S^T waits for that), then added into the accumulator with 16-byte
// atomic adds, which the warp does not wait for.
// ---------------------------------------------------------------------------
template <int D>
__device__ void bwd_dq(int wq, int lane, BwdBars* bars, uint32_t tmem, const BwdParams& p,
                       const BwdWork& w, unsigned int* err) {
    const volatile int* abort_flag = &bars->abort;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const int r = wq * 32 + lane;
    bool ok = true;
    for (int i = 0; i < w.n_tiles && ok; ++i) {
        ok = mbar_wait(smem_u32(&bars->dq_full), i & 1, abort_flag, 32);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[D];
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) tmem_ld32(tmem + cc + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[cc]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->dq_empty));
        const int hq = w.g * p.group + i / w.n_qt_cta;
        const int row = (w.qt_first + i % w.n_qt_cta) * kBT + r;
        if (row < p.Nq) {
            float4* dst = reinterpret_cast<float4*>(
                p.dq_acc + (((size_t)w.b * p.Hq + hq) * p.Nq_pad + (size_t)row) * D);
#pragma unroll
            for (int x = 0; x < D / 4; ++x)
                atomicAdd(dst + x, make_float4(__uint_as_float(v[4 * x]), __uint_as_float(v[4 * x + 1]),
                                               __uint_as_float(v[4 * x + 2]), __uint_as_float(v[4 * x + 3])));
        }
    }
    if (!ok) bwd_abort(bars, err);
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const __grid_constant__ CUtensorMap tdq, const BwdParams p, unsigned int* err) {
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
    const BwdWork w = bwd_work(p);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->qd_full[s]), 1);
            mbar_init(smem_u32(&bars->qd_empty[s]), 1 + 4);  // dK commit + 4 P/dS warps
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->p_full), 4);
        mbar_init(smem_u32(&bars->dq_full), 1);
        mbar_init(smem_u32(&bars->dq_empty), 4);
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tdq);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) bwd_producer<D>(&tq, &tk, &tv, &tdo, smem, bars, p, w, err);
    else if (warp == 1) bwd_mma<D>(smem, bars, tmem, w, err);
    else if (warp >= 4 && warp < 8) bwd_pds<D, OUT_F32>(warp & 3, lane, smem, bars, tmem, p, w, err);
    else if (warp >= 8) bwd_dq<D>(warp & 3, lane, bars, tmem, p, w, err);

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// prep / post
// ---------------------------------------------------------------------------
// One warp per padded query row: D = dO . O, lse2 = LSE log2(e) (padding:
// +inf, 0), and the row of the dQ accumulator set to zero.
template <int D>
__global__ void __launch_bounds__(256)
attn_bwd_prep_kernel(const void* __restrict__ o, int o_f32, const __nv_bfloat16* __restrict__ dout,
                     const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ dvec,
                     float* __restrict__ dq_acc, long long rows_pad, int Nq, int Nq_pad) {
    const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows_pad) return;
    const long long bh = r / Nq_pad;
    const int i = (int)(r - bh * Nq_pad);
    float4* acc = reinterpret_cast<float4*>(dq_acc + r * D);
    for (int c = lane; c < D / 4; c += 32) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
    if (i < Nq) {
        const size_t base = ((size_t)bh * Nq + i) * D;
        for (int c = lane; c < D; c += 32) {
            const float ov = o_f32 ? static_cast<const float*>(o)[base + c]
                                   : __bfloat162float(static_cast<const __nv_bfloat16*>(o)[base + c]);
            sum = fmaf(__bfloat162float(dout[base + c]), ov, sum);
        }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, s);
    if (lane == 0) {
        dvec[r] = i < Nq ? sum : 0.f;
        lse2[r] = i < Nq ? lse[(size_t)bh * Nq + i] * kBwdLog2e : INFINITY;
    }
}

template <bool OUT_F32>
__global__ void __launch_bounds__(256)
attn_bwd_post_kernel(const float* __restrict__ dq_acc, void* __restrict__ dq, long long n4, int Nq,
                     int Nq_pad, int d, float scale) {
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n4) return;
    const long long e = t * 4;                 // element of dq [B*Hq, Nq, d]
    const long long row = e / d;               // b*Hq*Nq + i
    const int c = (int)(e - row * d);
    const long long bh = row / Nq;
    const long long i = row - bh * Nq;
    const float4 v = *reinterpret_cast<const float4*>(dq_acc + ((bh * Nq_pad + i) * d + c));
    if constexpr (OUT_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(dq) + e) =
            make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    } else {
        uint2 pk;
        pk.x = pack_bf16x2(v.x * scale, v.y * scale);
        pk.y = pack_bf16x2(v.z * scale, v.w * scale);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dq) + e) = pk;
    }
}

template <int D, bool OUT_F32>
attn_status_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& p,
                           const void* o, int o_f32,
                           const void* dout, const float* lse, float* lse2, float* dvec,
                           void* dq, cudaStream_t stream, const DeviceInfo& dev) {
    using C = BwdCfg<D>;
    static int attr_set[64] = {0};
    if (dev.device < 64 && !attr_set[dev.device]) {
        if (cudaFuncSetAttribute(attn_bwd_kernel<D, OUT_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev.device] = 1;
    }
    const long long rows_pad = (long long)p.B * p.Hq * p.Nq_pad;
    attn_bwd_prep_kernel<D><<<(unsigned)((rows_pad + 7) / 8), 256, 0, stream>>>(
        o, o_f32, static_cast<const __nv_bfloat16*>(dout), lse, lse2, dvec, p.dq_acc, rows_pad,
        p.Nq, p.Nq_pad);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    const long long ctas = (long long)p.B * p.Hkv * p.n_kt;
    attn_bwd_kernel<D, OUT_F32><<<(unsigned)ctas, kBwdThreads, C::kSmemBytes, stream>>>(
        tq, tk, tv, tdo, tdq, p, dev.err_word);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    const long long n4 = (long long)p.B * p.Hq * p.Nq * D / 4;
    attn_bwd_post_kernel<OUT_F32><<<(unsigned)((n4 + 255) / 256), 256, 0, stream>>>(
        p.dq_acc, dq, n4, p.Nq, p.Nq_pad, D, p.scale);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int Nq, int d) {
    const size_t nq_pad = (size_t)((Nq + kBT - 1) / kBT) * kBT;
    const size_t rows = (size_t)B * Hq * nq_pad;
    return rows * (size_t)d * 4 + 2 * rows * 4;
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
        // L2 budget per section: a group's fp32 dQ accumulator rows, Q and dO
        // (bf16) of its query heads, and its K and V
        const long long per_group = (long long)p.group * p.Nq_pad * d * 4 +
                                    2ll * p.group * Nq * d * 2 + 2ll * Nk * d * 2;
        long long sgroups = (64ll << 20) / (per_group > 0 ? per_group : 1);
        if (sgroups < 1) sgroups = 1;
        if (sgroups > (long long)B * Hkv) sgroups = (long long)B * Hkv;
        p.sec_groups = (int)sgroups;
    }
    p.c = scale * kBwdLog2e;
    p.scale = scale;
    const size_t rows = (size_t)B * Hq * p.Nq_pad;
    p.dq_acc = static_cast<float*>(workspace);
    float* lse2 = p.dq_acc + rows * d;
    float* dvec = lse2 + rows;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dk = dk;
    p.dv = dv;
    if ((long long)B * Hkv * p.n_kt >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tq, tk, tv, tdo, tdq;
    attn_status_t st;
    if ((st = encode_tmap_bf16_3d(&tq, q, d, Nq, (long long)B * Hq, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tk, k, d, Nk, (long long)B * Hkv, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tv, v, d, Nk, (long long)B * Hkv, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_bf16_3d(&tdo, dout, d, Nq, (long long)B * Hq, kBT)) != ATTN_OK) return st;
    if ((st = encode_tmap_f32_sw128_3d(&tdq, p.dq_acc, d, p.Nq_pad, (long long)B * Hq, 32)) != ATTN_OK)
        return st;
    const int o_f32 = o_dtype == ATTN_OUT_F32;
    const bool g32 = grad_dtype == ATTN_OUT_F32;
    if (d == 128)
        return g32 ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tdq, p, o, o_f32, dout, lse, lse2, dvec, dq, stream, dev)
                   : launch_bwd_t<128, false>(tq, tk, tv, tdo, tdq, p, o, o_f32, dout, lse, lse2, dvec, dq, stream, dev);
    if (d == 64)
        return g32 ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tdq, p, o, o_f32, dout, lse, lse2, dvec, dq, stream, dev)
                   : launch_bwd_t<64, false>(tq, tk, tv, tdo, tdq, p, o, o_f32, dout, lse, lse2, dvec, dq, stream, dev);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace gb300
