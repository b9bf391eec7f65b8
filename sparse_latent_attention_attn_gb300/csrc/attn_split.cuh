// attn_split.cuh -- how the sparse_attn kernels share out their work: contiguous ranges of the
// flattened (work unit, index entry) space, one per persistent CTA or cluster, and the table of
// units that a range boundary cuts (merged afterwards by a combine kernel).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dsattn {
namespace split {

// Start of range c of the flattened entry space (unit t holds entries [t T, t T + T)).  The G
// ranges split a cost line evenly, on which each unit costs its T entries plus K: the fixed work
// of a segment (the epilogue, the next unit's q, refilling the row pipeline).  A range that starts
// more units then gets fewer entries, instead of finishing last.  A cut of the cost line inside a
// unit's K part falls on that unit's first entry; K = 0 is the even split of the entries.  The
// host guarantees G * ntok * (T + K) < 2^63, so the product is exact in 64 bits (a 128-bit
// division is a long software routine on the GPU).
__host__ __device__ __forceinline__ int64_t range_start(int64_t c, int64_t ntok, int64_t T, int64_t K, int64_t G) {
    const int64_t TK = T + K;
    if (TK <= 0 || G <= 0) return 0;
    const int64_t x = (int64_t)(((uint64_t)c * (uint64_t)(ntok * TK)) / (uint64_t)G);
    const int64_t tok = x / TK, r = x - tok * TK;
    return tok * T + (r > K ? r - K : 0);
}

// The work unit that position u of the unit order stands for.  With several queries per
// sequence (prefill) the cost of a query grows with its position (its window and its visible
// compressed rows fill up), so the order interleaves the units from both ends, 0, N-1, 1, N-2, ...:
// any contiguous range of positions then holds light and heavy units alike and the ranges' equal
// shares of the index entries become equal shares of the work.  The results do not depend on the
// order.
__host__ __device__ __forceinline__ int64_t unit_at(int64_t u, int64_t nunits, bool interleave) {
    return interleave ? ((u & 1) ? nunits - 1 - (u >> 1) : (u >> 1)) : u;
}

constexpr int kMaxCut = 160;   // cut units: at most one per range boundary, G <= SM count

// Number of ranges for a problem: stream-K over all gmax ranges when there are at least as many
// units as ranges; otherwise each unit gets the same number of ranges (split evenly), but no
// part shorter than two tiles of bn entries, and at most 32 parts (what a combine merges).
inline int64_t choose_ranges(int64_t ntok, int topk, int gmax, int bn) {
    if (ntok >= gmax) return gmax;
    int64_t k = gmax / ntok;
    const int64_t kmax = topk / (2 * bn) > 1 ? topk / (2 * bn) : 1;
    if (k > kmax) k = kmax;
    if (k > 32) k = 32;
    if (k < 1) k = 1;
    return ntok * k;
}

// K of range_start: seg when the ranges run several units each (stream-K); when the ranges split
// units evenly every part has the same fixed work, so the entries split evenly.
inline int64_t seg_cost(int64_t ntok, int64_t G, int64_t seg) { return G <= ntok ? seg : 0; }

// Whether some range boundary falls inside a unit (then partials and a combine are needed).
inline bool splits_units(int64_t ntok, int topk, int64_t G, int64_t K) {
    if (G <= 1 || topk == 0) return false;
    for (int64_t c = 1; c < G; ++c)
        if (range_start(c, ntok, topk, K, G) % topk != 0) return true;
    return false;
}

// The cut units of a launch: every unit that some range boundary falls inside, as
// {unit, first part (range), number of parts, slot bits}: bit i set when the unit is the last
// segment of part i (its partial is in that range's slot 1; slot 0 holds a range's first
// segment).  Returns the number of entries written to cut (at most kMaxCut), or -1 when a unit
// has more than 32 parts or there are too many cut units.
inline int cut_units(int64_t ntok, int64_t T, int64_t K, int64_t G, int4 *cut) {
    const int64_t E = ntok * T;
    auto start = [&](int64_t c) { return range_start(c, ntok, T, K, G); };
    int n = 0;
    int64_t last_tok = -1;
    for (int64_t c = 1; c < G; ++c) {
        const int64_t eb = start(c);
        if (eb % T == 0 || eb >= E) continue;
        const int64_t tok = eb / T;
        if (tok == last_tok) continue;               // already listed through an earlier boundary
        last_tok = tok;
        // parts: ranges that meet [tok T, tok T + T)
        int64_t kf = c - 1;
        while (kf > 0 && start(kf) > tok * T) --kf;
        int np = 0;
        uint32_t slots = 0;
        for (int64_t k = kf; k < G && start(k) < (tok + 1) * T; ++k) {
            if (start(k + 1) <= start(k)) continue;   // empty range
            if (np >= 32) return -1;
            if (start(k) / T != tok) slots |= 1u << np;          // the unit is k's last segment
            if (np == 0) kf = k;
            ++np;
        }
        if (n >= kMaxCut) return -1;
        cut[n++] = make_int4((int)tok, (int)kf, np, (int)slots);
    }
    return n;
}

}  // namespace split
}  // namespace dsattn
