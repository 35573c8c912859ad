// fwd_sched.h -- work decomposition of the fused forward, shared verbatim by the
// device kernel and the host-side exports (so the tests pin the code the
// kernel runs).
//
// A unit is (batch b, query head hq, m-block mb): 2 Q tiles of 128 rows,
// rows [256*mb, 256*mb + 256).  Both tiles stream the same K/V tiles, so K/V
// is loaded once per unit (lecture notes "Optimizing Attention for Modern
// Hardware", 3.1: Q-outer / KV-inner; "Flash Attention 3/4 notes", FA4
// section 1: two Q tiles per CTA).
//
// Order (lecture notes 4.5; FA4 notes section 3): query heads are grouped into
// sections whose K/V fit an L2 budget; sections run in order; inside a section
// the m-blocks run longest-first (causal) and, within one m-block rank, heads
// run in index order so GQA siblings (consecutive hq sharing a KV head) are
// adjacent.  The persistent CTAs take units from this list in order, each
// when it is ready for one (a device-side queue).
#pragma once

#include <algorithm>
#include <cstdint>
#include <functional>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#if defined(__CUDACC__)
#define GB300_HD __host__ __device__ __forceinline__
#else
#define GB300_HD inline
#endif

namespace gb300 {

constexpr int kTileM = 128;           // query rows per Q tile (tcgen05 M)
constexpr int kTileN = 128;           // keys per K/V tile
constexpr int kTilesPerUnit = 2;      // Q tiles per unit
constexpr int kUnitRows = kTileM * kTilesPerUnit;
// K/V bytes a section may span.  Non-causal units all cost the same, so a
// narrow section keeps the ~150 units in flight on few heads and their K/V
// resident in the near L2 partition.  Causal units differ in cost, and how
// well the longest-first order inside each section balances them depends on
// the section's width: a causal launch takes the narrowest of the candidate
// widths whose modelled makespan (causal_section_heads below) is within 1 %
// of the best; kL2SectionBytesCausal is the width used when no SM count is
// given.
constexpr long long kL2SectionBytesCausal = 64ll << 20;
constexpr long long kL2SectionBytesDense = 16ll << 20;
constexpr long long kCausalSectionCandidates[] = {8ll << 20, 16ll << 20, 32ll << 20, 64ll << 20,
                                                  128ll << 20};
// Fixed cost of a unit in the model, in KV steps (the epilogue and the next
// unit's first softmax, while the tensor cores idle; about 2.6 us against
// 1.4 us per step, measured).
constexpr double kUnitOverheadSteps = 2.0;

struct FwdShape {
    int B, Hq, Hkv, Nq, Nk, d, causal;
    int nmb;                 // m-blocks per head
    int heads_per_section;   // query heads per section (multiple of Hq/Hkv)
    long long units;         // B * Hq * nmb
};

// KV tiles needed by query rows [row0, row0 + rows): causal block skipping.
GB300_HD int kv_tiles_for_rows(int row0, int rows, int Nq, int Nk, int causal, int block) {
    if (rows <= 0 || Nk <= 0 || block <= 0) return 0;
    const int total = (Nk + block - 1) / block;
    if (!causal) return total;
    const long long last_key = (long long)row0 + rows - 1 + (long long)(Nk - Nq);
    if (last_key < 0) return 0;
    const long long t = last_key / block + 1;
    return t < total ? (int)t : total;
}

// Valid rows of Q tile t of m-block mb.
GB300_HD int tile_rows(int mb, int t, int Nq) {
    const int r0 = mb * kUnitRows + t * kTileM;
    const int r = Nq - r0;
    return r <= 0 ? 0 : (r < kTileM ? r : kTileM);
}

// KV tiles of Q tile t of m-block mb, for Nq query rows and Nk keys.
GB300_HD int tile_kv_count_len(int mb, int t, int Nq, int Nk, int causal) {
    return kv_tiles_for_rows(mb * kUnitRows + t * kTileM, tile_rows(mb, t, Nq), Nq, Nk, causal,
                             kTileN);
}

GB300_HD int tile_kv_count(int mb, int t, const FwdShape& s) {
    return tile_kv_count_len(mb, t, s.Nq, s.Nk, s.causal);
}

// Query heads per section for a K/V byte budget (a multiple of the GQA group).
inline int section_heads_for(int B, int Hq, int Hkv, int Nk, int d, long long budget) {
    const int group = Hq / Hkv;
    const long long kv_head_bytes = 2ll * Nk * d * 2;  // K and V, bf16
    long long kv_per_sec = budget / (kv_head_bytes > 0 ? kv_head_bytes : 1);
    if (kv_per_sec < 1) kv_per_sec = 1;
    long long hps = kv_per_sec * group;
    const long long all = (long long)B * Hq;
    if (hps > all) hps = all;
    return (int)hps;
}

// A unit covers unit_rows query rows: kUnitRows (two 128-row Q tiles, the
// d <= 128 kernels) or 128 (one Q tile, the d > 128 kernel).
inline FwdShape make_fwd_shape_sections(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                                        int heads_per_section, int unit_rows = kUnitRows) {
    FwdShape s;
    s.B = B; s.Hq = Hq; s.Hkv = Hkv; s.Nq = Nq; s.Nk = Nk; s.d = d; s.causal = causal;
    s.nmb = (Nq + unit_rows - 1) / unit_rows;
    s.heads_per_section = heads_per_section;
    s.units = (long long)B * Hq * s.nmb;  // the launcher rejects units >= 2^31
    return s;
}

GB300_HD void unit_of(const FwdShape& s, uint32_t i, int& bh, int& mb);

// Makespan, in KV steps, of the greedy list schedule of the units (lecture
// notes 4.5: each of num_sms workers takes the next unit of the list when it
// is free), a unit costing its KV steps plus kUnitOverheadSteps: for
// two-tile units the steps of the longer Q tile, for single-tile units
// (unit_rows 128, the d > 128 kernel) the tile's steps (128 keys each).
inline double list_makespan(const FwdShape& s, int num_sms, int unit_rows) {
    std::vector<double> load((size_t)num_sms, 0.0);  // a min-heap of worker loads
    for (long long i = 0; i < s.units; ++i) {
        int bh, mb;
        unit_of(s, (uint32_t)i, bh, mb);
        int steps;
        if (unit_rows == kUnitRows) {
            const int n0 = tile_kv_count(mb, 0, s), n1 = tile_kv_count(mb, 1, s);
            steps = n0 > n1 ? n0 : n1;
        } else {
            const int r0 = mb * kTileM;
            const int rows = s.Nq - r0 < kTileM ? s.Nq - r0 : kTileM;
            steps = kv_tiles_for_rows(r0, rows, s.Nq, s.Nk, s.causal, kTileN);
        }
        std::pop_heap(load.begin(), load.end(), std::greater<double>());
        load.back() += steps + kUnitOverheadSteps;
        std::push_heap(load.begin(), load.end(), std::greater<double>());
    }
    return *std::max_element(load.begin(), load.end());
}

// Heads per section of a causal launch on num_sms SMs: of the candidate K/V
// budgets, the narrowest whose modelled makespan is within 1 % of the best
// (narrower sections keep more of the K/V they stream in L2).  For the
// single-tile units of the d > 128 kernel the candidates start at 32 MiB:
// measured there (prefill shape at d = 256, causal) 16 MiB sections took
// 141.6 us against 135.8 us at 32 MiB and 137.2 us at 64 MiB, although the
// model ties them.  Cached per shape; shapes of more than 2^22 units keep the
// default width (the model's cost grows with the unit count).
inline int causal_section_heads(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_sms,
                                int unit_rows = kUnitRows) {
    const long long units = (long long)B * Hq * ((Nq + unit_rows - 1) / unit_rows);
    const int fallback = section_heads_for(B, Hq, Hkv, Nk, d, kL2SectionBytesCausal);
    if (num_sms < 1 || units > (1ll << 22)) return fallback;
    using Key = std::tuple<int, int, int, int, int, int, int, int>;
    static std::mutex mu;
    static std::map<Key, int> cache;
    const Key key{B, Hq, Hkv, Nq, Nk, d, num_sms, unit_rows};
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int heads[sizeof(kCausalSectionCandidates) / sizeof(kCausalSectionCandidates[0])];
    double span[sizeof(heads) / sizeof(heads[0])];
    double best = 0.0;
    int n = 0;
    for (long long budget : kCausalSectionCandidates) {
        if (unit_rows != kUnitRows && budget < (32ll << 20)) continue;
        const int h = section_heads_for(B, Hq, Hkv, Nk, d, budget);
        if (n > 0 && h == heads[n - 1]) continue;  // same list as the narrower budget
        heads[n] = h;
        span[n] = list_makespan(make_fwd_shape_sections(B, Hq, Hkv, Nq, Nk, d, 1, h, unit_rows),
                                num_sms, unit_rows);
        best = (n == 0 || span[n] < best) ? span[n] : best;
        ++n;
    }
    int choice = heads[n - 1];
    for (int i = 0; i < n; ++i)
        if (span[i] <= best * 1.01) { choice = heads[i]; break; }
    std::lock_guard<std::mutex> lk(mu);
    if (cache.size() > 256) cache.clear();
    cache[key] = choice;
    return choice;
}

// The launch shape.  num_sms > 0 lets causal launches choose their section
// width by the makespan model; 0 keeps the fixed budgets.
inline FwdShape make_fwd_shape(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                               int num_sms = 0, int unit_rows = kUnitRows) {
    const int hps = causal ? causal_section_heads(B, Hq, Hkv, Nq, Nk, d, num_sms, unit_rows)
                           : section_heads_for(B, Hq, Hkv, Nk, d, kL2SectionBytesDense);
    return make_fwd_shape_sections(B, Hq, Hkv, Nq, Nk, d, causal, hps, unit_rows);
}

// Unit index i (0 <= i < units < 2^31) -> (bh = b * Hq + hq, mb).  32-bit
// arithmetic keeps the device-side decode cheap; the host rejects shapes with
// 2^31 or more units.
GB300_HD void unit_of(const FwdShape& s, uint32_t i, int& bh, int& mb) {
    const uint32_t all = (uint32_t)s.B * (uint32_t)s.Hq;
    const uint32_t S = (uint32_t)s.heads_per_section;
    const uint32_t sec_units = S * (uint32_t)s.nmb;
    const uint32_t sec = i / sec_units;
    const uint32_t r = i - sec * sec_units;
    const uint32_t rest = all - sec * S;
    const uint32_t hs = rest < S ? rest : S;
    const uint32_t rank = r / hs;
    const uint32_t h_in = r - rank * hs;
    bh = (int)(sec * S + h_in);
    mb = s.causal ? (int)((uint32_t)s.nmb - 1u - rank) : (int)rank;
}

// Packed variable-length batches.  Sequence b holds rows [cu[b], cu[b+1]) of a
// packed [total, H, d] array.  Its tensor maps add two dimensions so that the
// hardware's bounds check stops exactly at each sequence's end (loads past it
// read zeros, stores past it are dropped): element (c, h, r, e, f) lies at
//   base + c*es + h*d*es + (r + e)*rs + f*(2^34 - rs)        (mod 2^64),
// rs the row stride.  Row `row` of a sequence starting at s with length L uses
// r = W - L + row, e = s + L, f = W with W = 2^30: the f term is
// W*2^34 - W*rs = 2^64 - W*rs, so the address is base + (s + row)*rs, and
// r < W (the extent of r) holds exactly when row < L.
constexpr int kRaggedWindow = 1 << 30;     // W: extent of r, and the f coordinate
constexpr unsigned kRaggedOuterExtent = 0x7FFFFFFFu;  // extents of e and f (> W)

// Tail split.  Without causal masking every unit costs the same, so a unit
// count just above a multiple of the SM count leaves most CTAs idle in the
// last round (512 units on 152 SMs: 56 CTAs run a 4th unit), and fewer units
// than SMs leave SMs idle throughout.  The units of that last round ("tail"
// units) are then cut along the KV range into `parts` pieces that run on
// otherwise idle CTAs; each piece keeps its own (m, l) and
// O, and the last piece to finish merges them (lecture notes 6.1: split-KV
// pieces merged by the rescaling rule of 2.2, exact for any number of pieces).  Causal launches are not split: their units differ in
// cost and the longest-first order already fills the last round.
constexpr int kMaxSplitParts = 8;
constexpr int kMaxSplitUnits = 255;

struct FwdSplit {
    int n_full;   // units run whole: list positions [0, n_full)
    int n_split;  // tail units run in parts: list positions [n_full, n_full + n_split)
    int parts;    // pieces per tail unit (1 when nothing is split)
};

GB300_HD FwdSplit plan_tail_split(const FwdShape& s, int num_sms) {
    FwdSplit r;
    r.n_full = (int)s.units; r.n_split = 0; r.parts = 1;
    if (s.causal || num_sms < 2 || s.units < 1) return r;
    const long long tail = s.units % num_sms;
    if (tail == 0 || tail > kMaxSplitUnits) return r;
    long long parts = num_sms / tail;               // all pieces in one round
    const int n = kv_tiles_for_rows(0, 1, s.Nq, s.Nk, 0, kTileN);  // KV tiles per unit
    if (parts > n) parts = n;
    if (parts > kMaxSplitParts) parts = kMaxSplitParts;
    if (parts < 2) return r;
    r.n_full = (int)(s.units - tail);
    r.n_split = (int)tail;
    r.parts = (int)parts;
    return r;
}

GB300_HD uint32_t split_items(const FwdSplit& sp) {
    return (uint32_t)sp.n_full + (uint32_t)sp.n_split * (uint32_t)sp.parts;
}

// Work item -> unit (list position) and piece (-1: the whole unit).
GB300_HD void item_of(const FwdSplit& sp, uint32_t item, uint32_t& unit, int& part) {
    if (item < (uint32_t)sp.n_full) { unit = item; part = -1; return; }
    const uint32_t r = item - (uint32_t)sp.n_full;
    const uint32_t k = r / (uint32_t)sp.parts;
    unit = (uint32_t)sp.n_full + k;
    part = (int)(r - k * (uint32_t)sp.parts);
}

// KV tiles [j0, j1) of piece `part` of a unit with n KV tiles.
GB300_HD void part_range(int n, int parts, int part, int& j0, int& j1) {
    if (part < 0) { j0 = 0; j1 = n; return; }
    j0 = (int)((long long)part * n / parts);
    j1 = (int)((long long)(part + 1) * n / parts);
}

}  // namespace gb300
