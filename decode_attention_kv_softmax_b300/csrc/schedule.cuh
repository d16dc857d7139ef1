// Balanced split-KV work schedule shared by the decode kernels.
//
// The KV of every sequence b is cut into tiles of 64 tokens (one page);
// sequence b contributes `upb` work units (KV heads x head chunks for GQA,
// one unit per sequence for MLA) of ntiles(b) = ceil(len_b / 64) tiles each.
// All tiles are laid end to end (b-major, then unit, then tile) and W work
// items take equal contiguous shares: item w covers tiles
// [floor(T w / W), floor(T (w+1) / W)).  This is flash-decoding's split of
// the sequence ([ARG] "attention-variants-and-kv-cache" §五.2, last
// paragraph) with the cut points chosen so that every CTA streams the same
// number of bytes whatever the length mix.  A unit whose tiles fall into one
// item is finished by that item; a unit cut by item boundaries leaves one
// normalised partial per piece, and the last piece to finish merges them.
//
// Partial slots: item w owns slots 2w (the piece holding the item's first
// tile) and 2w+1 (the piece holding its last tile, when that is a different
// unit).  Only these two pieces of an item can be incomplete units.
//
// Unit start cost.  Starting a unit costs a CTA more than a tile where the
// switch is slow (the MLA kernel loads a new Q into TMEM and flushes O at
// every switch), so the cut points can be chosen on a cost axis instead of
// the tile axis: unit u = b * upb + j (empty units included) occupies
// [u c + first tile of u, ...), i.e. c cost units of start overhead and then
// one per tile, and the cost position of tile t of unit u is t + c (u + 1).
// With total cost C = T + c B upb, item w covers the cost range
// [floor(C w / W), floor(C (w+1) / W)) and starts at the first tile whose
// cost position lies in it.  Cost positions grow strictly with t, so the
// items still cover consecutive tile ranges (an item can be empty when a cut
// lands in overhead) and a unit's pieces still sit in consecutive items;
// c = 0 is the plain tile split above.
#pragma once

#include "common.cuh"

namespace kvdec {

constexpr int kTileTokens = 64;

struct TileSchedule {
    const int* cum;  // shared memory, [B+1]: cum[b] = sum_{b'<b} ntiles(b')
    int B;
    int upb;
    long long T;  // total tiles
    int W;        // work items (>= 1)
    int c = 0;    // start cost of a unit, in tiles

    KVDEC_HDINL int ntiles(int b) const { return cum[b + 1] - cum[b]; }
    KVDEC_HDINL long long total_cost() const { return T + (long long)c * B * upb; }
    // cost position of tile t, which is tile lt of unit (b, j)
    KVDEC_HDINL long long cost_of(int b, int j, long long t) const {
        return t + (long long)c * ((long long)b * upb + j + 1);
    }
    // first tile of item w (T for w = W)
    KVDEC_HDINL long long item_begin(int w) const {
        if (c == 0) return T * (long long)w / W;
        const long long C = total_cost();
        const long long X = C * (long long)w / W;   // the item's first cost position
        if (X >= C) return T;
        // the last sequence whose first unit starts (overhead included) at or before X
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long long)cum[mid] * upb + (long long)c * mid * upb <= X) lo = mid;
            else hi = mid;
        }
        const int b = lo, nt = ntiles(b);
        const long long s0 = (long long)cum[b] * upb + (long long)c * b * upb;
        long long j = (X - s0) / (nt + c);
        if (j > upb - 1) j = upb - 1;
        const long long off = X - s0 - j * (nt + c);   // into unit (b, j): c of overhead, then its tiles
        const long long first = (long long)cum[b] * upb + j * nt;
        if (off <= c) return first;
        const long long lt = off - c;
        return first + (lt < nt ? lt : nt);   // past the unit's tiles: the next unit's first tile
    }
    // the item holding tile t of unit (b, j)
    KVDEC_HDINL int item_of_in(int b, int j, long long t) const {
        const long long x = cost_of(b, j, t);
        return (int)(((x + 1) * (long long)W - 1) / total_cost());
    }
    KVDEC_HDINL long long unit_begin(int b, int j) const {
        return (long long)cum[b] * upb + (long long)j * ntiles(b);
    }
    // the item holding global tile t
    KVDEC_HDINL int item_of(long long t) const {
        if (c == 0) return (int)(((t + 1) * (long long)W - 1) / T);
        int b, j, lt;
        locate(t, b, j, lt);
        return item_of_in(b, j, t);
    }
    // (b, j, lt) of global tile t, 0 <= t < T
    KVDEC_HDINL void locate(long long t, int& b, int& j, int& lt) const {
        int lo = 0, hi = B;  // cum[lo]*upb <= t < cum[hi]*upb
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long long)cum[mid] * upb <= t) lo = mid;
            else hi = mid;
        }
        b = lo;
        const long long off = t - (long long)cum[b] * upb;
        const int nt = ntiles(b);
        j = (int)(off / nt);
        lt = (int)(off % nt);
    }
    // number of pieces unit (b, j) is cut into, and the slot of piece s
    KVDEC_HDINL int num_pieces(int b, int j) const {
        const long long t0 = unit_begin(b, j);
        return item_of_in(b, j, t0 + ntiles(b) - 1) - item_of_in(b, j, t0) + 1;
    }
    // first item holding unit (b, j) and the slot kind of its first piece;
    // piece s >= 1 lives in slot 2 * (w0 + s)
    KVDEC_HDINL void first_piece(int b, int j, int& w0, int& kind0) const {
        const long long t0 = unit_begin(b, j);
        w0 = item_of_in(b, j, t0);
        kind0 = (t0 != item_begin(w0)) ? 1 : 0;
    }
    KVDEC_HDINL int piece_slot(int b, int j, int s) const {
        const long long t0 = unit_begin(b, j);
        const int w0 = item_of_in(b, j, t0);
        const int kind = (s == 0 && t0 != item_begin(w0)) ? 1 : 0;
        return 2 * (w0 + s) + kind;
    }
};

// Walks global tiles in order, tracking the unit and the tile inside it.
struct TileCursor {
    int b, j, lt, nt;
    KVDEC_HDINL void start(const TileSchedule& S, long long t) {
        S.locate(t, b, j, lt);
        nt = S.ntiles(b);
    }
    KVDEC_HDINL void advance(const TileSchedule& S) {
        if (++lt < nt) return;
        lt = 0;
        if (++j < S.upb) return;
        j = 0;
        do {
            ++b;
        } while (b < S.B && S.ntiles(b) == 0);
        nt = (b < S.B) ? S.ntiles(b) : 0;
    }
};

// Clamp a sequence length to [0, cap], reporting out-of-range values.
KVDEC_DEVINL int clamp_len(int len, int cap, uint32_t* err) {
    if (len < 0) {
        report(err, KVDEC_DEVERR_SEQLEN);
        return 0;
    }
    if (len > cap) {
        report(err, KVDEC_DEVERR_SEQLEN);
        return cap;
    }
    return len;
}

// Tokens one decode step reads from the cache: every one of the sequence's
// len tokens, or with a sliding window of w tokens kept in a ring cache of w
// slots ([ARG] "attention-variants-and-kv-cache" §五.3) the min(len, w)
// slots that hold the last w positions (softmax does not depend on their
// order).  Clamped to the capacity like the plain length.
KVDEC_DEVINL int read_len(int len, int window, int cap, uint32_t* err) {
    if (window > 0 && len > window) len = window;
    return clamp_len(len, cap, err);
}

// Block-wide: cum[0..B] from seqlens (read_len of each).  `scratch` holds
// blockDim.x ints.  Each thread sums a contiguous chunk of
// sequences, warp 0 scans the per-thread sums with shuffles, and each thread
// writes its chunk's prefix.  Ends with __syncthreads().
KVDEC_DEVINL void build_cum(int* cum, int* scratch, const int32_t* seqlens, int B, int cap,
                            uint32_t* err, int window = 0) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int chunk = (B + nth - 1) / nth;
    const int lo = min(B, tid * chunk), hi = min(B, lo + chunk);
    int sum = 0;
    for (int b = lo; b < hi; ++b) {
        const int len = read_len(__ldg(seqlens + b), window, cap, blockIdx.x == 0 ? err : nullptr);
        sum += (len + kTileTokens - 1) / kTileTokens;
    }
    scratch[tid] = sum;
    __syncthreads();
    if (tid < 32) {
        // lane l owns scratch[l*per .. l*per + per), any block size
        const int per = (nth + 31) / 32;
        const int lo_i = min(nth, tid * per), hi_i = min(nth, lo_i + per);
        int tot = 0;
        for (int idx = lo_i; idx < hi_i; ++idx) tot += scratch[idx];
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (tid >= off) incl += u;
        }
        int run = incl - tot;
        for (int idx = lo_i; idx < hi_i; ++idx) {
            const int v = scratch[idx];
            scratch[idx] = run;
            run += v;
        }
        if (tid == 31) cum[B] = incl;
    }
    __syncthreads();
    int run = scratch[tid];
    for (int b = lo; b < hi; ++b) {
        cum[b] = run;
        const int len = read_len(__ldg(seqlens + b), window, cap, nullptr);
        run += (len + kTileTokens - 1) / kTileTokens;
    }
    __syncthreads();
}

// Counts the arrival of one piece of a split unit and tells the caller
// whether it was the last one.  A counter word holds (epoch << 32 | count);
// a word from another call (any other epoch, including leftovers of an
// aborted call or unrelated bytes of a reused workspace) counts as zero, so
// the workspace needs no initialisation.  The last arriver stores 0, which
// keeps replays of a captured launch (same epoch) correct as well.
KVDEC_DEVINL bool arrive_piece(unsigned long long* ctr, uint32_t epoch, uint32_t npieces) {
    unsigned long long seen = *reinterpret_cast<volatile unsigned long long*>(ctr);
    uint32_t count;
    while (true) {
        count = ((uint32_t)(seen >> 32) == epoch) ? (uint32_t)seen : 0u;
        const unsigned long long next = ((unsigned long long)epoch << 32) | (count + 1u);
        const unsigned long long prev = atomicCAS(ctr, seen, next);
        if (prev == seen) break;
        seen = prev;
    }
    return count + 1u == npieces;
}

// Number of work items actually used: at most `grid`, and at least
// `min_tiles` tiles per item on average.
KVDEC_HDINL int effective_items(long long T, int grid, int min_tiles) {
    long long w = (T + min_tiles - 1) / min_tiles;
    if (w < 1) w = 1;
    if (w > grid) w = grid;
    return (int)w;
}

}  // namespace kvdec
