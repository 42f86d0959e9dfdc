// k2_items.h -- the work items of the prefill attention kernels (host and
// device code; nothing here needs the CUDA runtime).
//
// An item is one 128-row query block of one sequence for `hpi` query heads of
// one kv head.  Items are listed heaviest first: by level (the query block
// qb, highest first), then by sequence among those with a block at that
// level, then kv head, then head group (`npairs` per kv head).  A persistent
// grid deals them out in snake order: round k gives worker c item
// k G + c for even k and k G + G - 1 - c for odd k (G workers).
//
// Every role of a worker walks its items in increasing index order, so a
// walk keeps the level it is at (the index of the level's first item and its
// item count) and enters each level once: an item costs a few comparisons,
// not a pass over every level above it.
#pragma once

#ifdef __CUDACC__
#define QA_ITEMS_FN __host__ __device__ __forceinline__
#else
#define QA_ITEMS_FN inline
#endif

namespace qa {

struct K2Walk {
    int lvl = -1;  // level of the last item decoded (-1: not started)
    int base = 0;  // index of the level's first item
    int cnt = 0;   // items at the level
};

// Geometry of one work item, the same in every role.
struct K2Item {
    int b, kvh, qb;   // sequence, kv head, query block
    int h0;           // first query head of the item
    int L;            // new tokens of the sequence
    int qmin;         // position of the block's row 0
    int j0, nkv;      // first key tile and number of key tiles
    int jmask;        // key tiles from this one on may hold keys past a row's position
    int row0;         // row of the block's row 0 in q' / out
};

// The snake order: worker c's k-th item index among G workers.
QA_ITEMS_FN int k2_snake_index(int k, int G, int c) { return k * G + ((k & 1) ? G - 1 - c : c); }

// Sequences with a query block at level lvl (len > 128 lvl).  P: the launch
// parameters (nseq, len[], start[], cu[], Hkv, G, npairs, hpi, max_qblocks,
// nitems, window).
template <class P>
QA_ITEMS_FN int k2_level_seqs(const P &p, int lvl) {
    constexpr int n = static_cast<int>(sizeof(p.len) / sizeof(p.len[0]));
    int e = 0;
#pragma unroll
    for (int s = 0; s < n; ++s) e += (s < p.nseq && p.len[s] > lvl * 128) ? 1 : 0;
    return e;
}

// Item idx (never below the walk's last item) as sequence, kv head, head
// group and query block; false past the last item.
template <class P>
QA_ITEMS_FN bool k2_decode_item(const P &p, int idx, K2Walk &w, int &b, int &kvh, int &pair, int &qb) {
    constexpr int n = static_cast<int>(sizeof(p.len) / sizeof(p.len[0]));
    const int per_seq = p.Hkv * p.npairs;
    if (w.lvl < 0) {
        w.lvl = p.max_qblocks - 1;
        w.base = 0;
        w.cnt = k2_level_seqs(p, w.lvl) * per_seq;
    }
    while (idx >= w.base + w.cnt) {
        w.base += w.cnt;
        if (--w.lvl < 0) return false;
        w.cnt = k2_level_seqs(p, w.lvl) * per_seq;
    }
    const int off = idx - w.base;
    int which = off / per_seq;
    const int rem = off - which * per_seq;
    b = 0;
#pragma unroll
    for (int s = 0; s < n; ++s) {
        const bool has = s < p.nseq && p.len[s] > w.lvl * 128;
        if (has && which == 0) b = s;
        which -= has ? 1 : 0;
    }
    kvh = rem / p.npairs;
    pair = rem - kvh * p.npairs;
    qb = w.lvl;
    return true;
}

// Item idx with its geometry (false past the last; idx never below the
// walk's last call).  With a window of W keys, row i sees keys
// max(0, i + 1 - W) .. i; without, keys 0 .. i.
template <bool kWindow, class P>
QA_ITEMS_FN bool k2_item_at(const P &p, int idx, K2Walk &w, K2Item &it) {
    if (idx >= p.nitems) return false;
    int pair = 0;
    if (!k2_decode_item(p, idx, w, it.b, it.kvh, pair, it.qb)) return false;
    it.h0 = it.kvh * p.G + p.hpi * pair;
    it.L = p.len[it.b];
    it.qmin = p.start[it.b] + it.qb * 128;
    const int lo = it.qmin + 1 - p.window;
    it.j0 = kWindow ? (lo > 0 ? lo : 0) / 128 : 0;
    const int last_row = it.L - 1 - it.qb * 128;
    it.nkv = (it.qmin + (last_row < 127 ? last_row : 127)) / 128 + 1 - it.j0;
    it.jmask = it.qmin / 128;
    it.row0 = p.cu[it.b] + it.qb * 128;
    return true;
}

}  // namespace qa
