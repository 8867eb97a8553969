// Work items of the expert phase.  The routed pairs of a layer are grouped per
// expert (perm order: each expert's pairs in (token, slot) order) and cut into
// chunks of at most 8 pairs (blocks routed through the workspace: 32 pairs with 4 E2M1
// terms per activation, or 16 with 8, so that a chunk fills the MMA's 128 activation
// rows).  For every chunk there are I/128 gate/up items (a
// 128-row block of the gate and of the up matrix over all of K = H) and H/256 down
// items (a 256-row block of the down matrix over all of K = I).  Within an expert the
// items are ordered row block major, chunk minor: the chunks that read the same
// weight rows are claimed one after another, so those rows are streamed from HBM
// once and served from L2 to the other chunks.
#pragma once

#include "common.cuh"
#include "route.cuh"

namespace moe {

constexpr int kTmaRows = 128;   // rows per gate/up item (of each of the two matrices)
constexpr int kDownRows = 256;  // rows per down item
constexpr int kTmaTok = 8;      // pairs per chunk (8 E2M1 terms per activation)
// blocks routed through the workspace: chunks fill the MMA's 128 activation rows
constexpr int kDenseTok = 32;   // pairs per chunk of the dense operand (4 terms per activation)
constexpr int kWideTok = 16;    // pairs per chunk with 8 terms per activation
constexpr int kMaxChunk = 16;   // words of pair ids in a record

enum : int { kItemGateUp = 0, kItemDown = 1 };

// Work item code: bit 30 = kind, bits 20..29 = row block, bits 11..19 = chunk of the
// expert, bits 0..10 = index into the routed-expert list.
__host__ __device__ __forceinline__ int item_code(int kind, int rb, int tc, int a) {
    return (kind << 30) | (rb << 20) | (tc << 11) | a;
}

// One work item as the producer reads it (96 bytes).
struct __align__(16) ItemRec {
    int code;            // item_code(kind, rb, tc, a)
    int e;               // expert id
    int beg;             // first position of the chunk's pairs in perm
    int ntok;            // pairs in the chunk (1..8; blocks routed through the workspace: 1..32)
    int tok[kMaxChunk];  // gate/up items: token of each pair; down items: pair id (t*k + j);
                         // blocks routed through the workspace: 16-bit halves, pair slots
                         // 2q and 2q + 1 in word q
    int chunk;           // chunk index within the layer
    int pad[3];          // pad[0]: chunks of the expert (the items of one row block are adjacent)
};

// Routing state of one layer kept in shared memory by every CTA when the verify
// block is small (T*k <= 64 pairs): the work items are derived from it directly.
constexpr int kRtMaxPairs = 64;
struct RouteTable {
    int n_active, n_chunks, pad0, pad1;
    int e[kRtMaxPairs];        // per routed expert (ascending id): expert id
    int beg[kRtMaxPairs];      // first position in perm
    int cnt[kRtMaxPairs];      // pairs routed to it
    int chunk0[kRtMaxPairs];   // index of its first chunk
    int tok[kRtMaxPairs];      // per perm position: token
    int pair[kRtMaxPairs];     // per perm position: pair id t*k + j
    int idx[kRtMaxPairs];      // per pair t*k + j: routed expert
    float gate[kRtMaxPairs];   // per pair t*k + j: gate
    float tscale[kRtMaxPairs]; // per token (residual stack): 1 / rms of its residual
    const float* tscale_g;     // the same factors in global memory [T] (blocks routed through the workspace)
};

// Per-forward work list (workspace).
struct WorkList {
    ItemRec* items;    // all gate/up items, then all down items
    int* n_items;      // [0] = total, [1] = number of gate/up items
    int* queue;        // next item to claim (zero at the start of the phase)
    int* done;         // [chunks] gate/up items finished per chunk (zero at the start)
    int* abort;        // set when any wait times out
    int* chunk0;       // [n_active + 1] first chunk of each routed expert, then the total (larger blocks)
};

// Item idx of the phase, from the routing table (rbu / rbd: row blocks of gate/up and down).
__device__ __forceinline__ ItemRec table_item(const RouteTable* rt, int idx, int rbu, int rbd) {
    const int n_gu = rt->n_chunks * rbu;
    const bool down = idx >= n_gu;
    const int j = down ? idx - n_gu : idx;
    const int nrb = down ? rbd : rbu;
    int lo = 0, hi = rt->n_active - 1;   // the routed expert whose items contain j
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (rt->chunk0[mid] * nrb <= j) lo = mid; else hi = mid - 1;
    }
    const int nch = (rt->cnt[lo] + kTmaTok - 1) / kTmaTok;
    const int rr = j - rt->chunk0[lo] * nrb, rbi = rr / nch, tc = rr % nch;   // row block major, chunk minor
    const int chunk = rt->chunk0[lo] + tc;
    ItemRec r;
    r.code = item_code(down ? kItemDown : kItemGateUp, rbi, tc, lo);
    r.e = rt->e[lo];
    r.beg = rt->beg[lo] + tc * kTmaTok;
    r.ntok = min(kTmaTok, rt->cnt[lo] - tc * kTmaTok);
#pragma unroll
    for (int q = 0; q < kMaxChunk; ++q) r.tok[q] = q < r.ntok ? (down ? rt->pair[r.beg + q] : rt->tok[r.beg + q]) : 0;
    r.chunk = chunk;
    r.pad[0] = nch;
    r.pad[1] = r.pad[2] = 0;
    return r;
}

// A record written by another CTA of the same launch: read from L2.
__device__ __forceinline__ ItemRec load_item(const ItemRec* src) {
    ItemRec r;
    const int4* s = reinterpret_cast<const int4*>(src);
    int4* d = reinterpret_cast<int4*>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(ItemRec) / 16); ++i) d[i] = __ldcg(s + i);
    return r;
}

// Builds the work list of one layer from the grouping (one block of 1024 threads):
// chunk offsets by a scan over the routed experts, then every item's full record
// (gate/up items first).  Dynamic shared memory: T*k ints (the perm).
__global__ void __launch_bounds__(1024) build_items_kernel(RouteBufs rb, int H, int I, int k, WorkList wl, int T) {
    __shared__ int s_gu[kMaxExperts + 1];
    __shared__ int s_act[kMaxExperts], s_beg[kMaxExperts], s_cnt[kMaxExperts];
    __shared__ int s_scan[64];
    extern __shared__ int s_perm[];   // [T * k] pair id of each perm position
    const int n_active = rb.active[0];
    const int rbu = I / kTmaRows, rbd = H / kDownRows;
    const int a = threadIdx.x;
    int chunks = 0;
    if (a < n_active) {
        const int e = rb.active[1 + a];
        s_act[a] = e;
        s_beg[a] = rb.offsets[e];
        s_cnt[a] = rb.counts[e];
        chunks = (s_cnt[a] + kTmaTok - 1) / kTmaTok;
    }
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) s_perm[i] = rb.perm[i];
    const int off = block_excl_scan_1024(chunks, s_scan);
    const int total_chunks = s_scan[32];
    if (a < n_active) s_gu[a] = off;
    for (int c = threadIdx.x; c < total_chunks; c += blockDim.x) wl.done[c] = 0;
    __syncthreads();
    const int n_gu = total_chunks * rbu;
    if (threadIdx.x == 0) {
        wl.n_items[0] = n_gu + total_chunks * rbd;
        wl.n_items[1] = n_gu;
        *wl.queue = 0;
        *wl.abort = 0;
    }
    const int total = total_chunks * (rbu + rbd);
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const bool down = i >= n_gu;
        const int j = down ? i - n_gu : i;
        const int nrb = down ? rbd : rbu;
        int lo = 0, hi = n_active - 1;          // the routed expert whose items contain j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_gu[mid] * nrb <= j) lo = mid; else hi = mid - 1;
        }
        const int aa = lo;
        const int nch = (s_cnt[aa] + kTmaTok - 1) / kTmaTok;
        const int rr = j - s_gu[aa] * nrb, rbi = rr / nch, tc = rr % nch;   // row block major, chunk minor
        const int chunk = s_gu[aa] + tc;
        ItemRec r;
        r.code = item_code(down ? kItemDown : kItemGateUp, rbi, tc, aa);
        r.e = s_act[aa];
        r.beg = s_beg[aa] + tc * kTmaTok;
        r.ntok = min(kTmaTok, s_cnt[aa] - tc * kTmaTok);
#pragma unroll
        for (int q = 0; q < kMaxChunk; ++q) r.tok[q] = q < r.ntok ? (down ? s_perm[r.beg + q] : s_perm[r.beg + q] / k) : 0;
        r.chunk = chunk;
        r.pad[0] = nch;
        r.pad[1] = r.pad[2] = 0;
        wl.items[i] = r;
    }
}

}  // namespace moe
