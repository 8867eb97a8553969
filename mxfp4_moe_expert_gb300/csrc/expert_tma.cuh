// Warp-specialised expert FFN for the skinny regime (a handful of tokens per
// expert), fed by TMA.
//
// The expert weights are the layer's bytes: each routed expert's gate, up and
// down matrices are streamed from HBM exactly once per verify block ("MiMo x
// TileRT", 万亿参数推理为什么特别难: decode speed = bandwidth / bytes read).
// One persistent CTA per SM pulls work items from a queue.  An item is a
// 128-row tile of one expert's gate+up (all of K = H) or down (all of K = I)
// matrix for up to 8 of its tokens.  Inside the CTA ("MiMo 把 1T 模型推到每秒千
// token", persistent engine kernel and warp specialization section: data-movement
// warps prefetch the next tile while compute warps work on the current one):
//   - warp 8 (producer) claims items and streams their K-stages with TMA into a
//     ring of shared-memory slots: two 128-byte-swizzled nibble boxes
//     [128 rows x 128 B], the E8M0 scale box [128 rows x 16 B] and the f16
//     activation chunks of the item's tokens;
//   - warps 0..7 (consumers): warp w owns rows 32(w%4)..+31 of the item for the
//     K half w/4 of every stage.  They decode E2M1 code pairs straight from the
//     swizzled tile into f16 MMA fragments with the hardware pair conversion and
//     multiply them with the tokens' f16 activations on the tensor cores
//     (mma.sync m16n8k16, exact products, fp32 accumulation; N = 8 covers the
//     item's tokens).  The K order inside each 16-wide MMA is permuted so that
//     every MMA stays inside one 32-element MX block; each block's fp32 result is
//     then scaled by its 2^(S-127).
// Gate/up items end with SwiGLU and store h in f16 with a power-of-two scale per
// (pair, 128-row segment); down items wait (bounded) until every gate/up item of
// their expert has published h, and store fp32 per-pair partial outputs.
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "route.cuh"

namespace moe {

constexpr int kTmaRows = 128;        // rows per item
constexpr int kTmaKC = 512;          // K elements per stage
constexpr int kTmaTok = 8;           // tokens per item
constexpr int kTmaStages = 5;        // ring slots
#ifndef MOE_TMA_CONSUMER_WARPS
#define MOE_TMA_CONSUMER_WARPS 16
#endif
constexpr int kTmaConsumerWarps = MOE_TMA_CONSUMER_WARPS;   // 8: two 16-row tiles per warp; 16: one
constexpr int kTmaTiles = 16 / kTmaConsumerWarps;            // 16-row MMA tiles per consumer warp
constexpr int kTmaRowGroups = kTmaConsumerWarps / 2;         // warps per K half
constexpr int kTmaThreads = (kTmaConsumerWarps + 1) * 32;
constexpr int kSlotNib = 2 * kTmaRows * 128;               // 32 KB
constexpr int kSlotScale = kTmaRows * 16;                  // 2 KB
constexpr int kActStride = kTmaKC * 2 + 64;                // bytes per token row (padding: conflict-free B loads)
constexpr int kSlotAct = kTmaTok * kActStride;             // 8.5 KB
constexpr int kSlotAux = 512;                              // down items: h segment scales [8 tok][4]
constexpr int kSlotBytes = kSlotNib + kSlotScale + kSlotAct + kSlotAux;  // 43 KB, multiple of 1024
static_assert(kSlotBytes % 1024 == 0, "slots hold 1024-byte-aligned swizzled boxes");
constexpr int kEpiBytes = kTmaRows * kTmaTok * 2 * 4;      // K-half exchange: 8 KB
constexpr int kTmaSmemBytes =
    1024 /*align slack*/ + kTmaStages * kSlotBytes + kEpiBytes + 2048 /*barriers, slot meta, routing table*/;
static_assert(kTmaSmemBytes <= 232448, "shared memory of the expert kernel");
static_assert(8 * (2 * kTmaStages + 1) + sizeof(int) * 8 * kTmaStages + sizeof(int) * (4 + 6 * 64) <= 2048,
              "barriers, slot metadata and routing table fit their region");

enum : int { kItemGateUp = 0, kItemDown = 1 };

// Work item code: bit 30 = kind, bits 20..29 = row block, bits 11..19 = token chunk,
// bits 0..10 = index into the active-expert list.
__host__ __device__ __forceinline__ int item_code(int kind, int rb, int tc, int a) {
    return (kind << 30) | (rb << 20) | (tc << 11) | a;
}

struct TmaMaps {
    CUtensorMap gate_q, up_q, down_q;   // uint8 2D [rows, K/2], box {128 B, 128 rows}, 128B swizzle
    CUtensorMap gate_s, up_s, down_s;   // uint8 2D [rows, K/32], box {16 B, 128 rows}
};

// One work item, as the producer reads it (64 bytes): everything it needs to
// issue the item's copies without further dependent loads.
struct __align__(16) ItemRec {
    int code;          // item_code(kind, rb, tc, a)
    int e;             // expert id
    int beg;           // first position of the item's pairs in perm
    int ntok;          // pairs in the item (1..8)
    int tok[kTmaTok];  // gate/up items: token of each pair; down items: pair id (t*k + j)
    int pad[4];
};

// Routing state of one layer kept in shared memory by every CTA when the verify
// block is small (T*k <= 64 pairs): the work items are derived from it directly.
constexpr int kRtMaxPairs = 64;
struct RouteTable {
    int n_active, n_chunks, pad0, pad1;
    int e[kRtMaxPairs];        // per routed expert (ascending id): expert id
    int beg[kRtMaxPairs];      // first position in perm
    int cnt[kRtMaxPairs];      // pairs routed to it
    int chunk0[kRtMaxPairs];   // index of its first chunk of <= 8 pairs
    int tok[kRtMaxPairs];      // per perm position: token
    int pair[kRtMaxPairs];     // per perm position: pair id t*k + j
};

// Per-forward work list and synchronisation words (workspace, zeroed per layer).
struct WorkList {
    ItemRec* items;    // all gate/up items, then all down items (unused with a routing table)
    int* n_items;      // [0] = total, [1] = number of gate/up items
    int* queue;        // next item to claim (zero at the start of the phase)
    int* done;         // [E] gate/up items finished, per active-expert index (zero at the start)
    int* need;         // [E] gate/up items per active-expert index
    int* abort;        // set when any wait times out
};

struct ExpertArgs {
    int H, I, k, layer;
    const __half* act16;     // [T, H] f16 activations, x * 2^-p (p per token and 128-wide segment)
    const float* act_fac;    // [T, H / 128] 2^p of each segment
    __half* h16;             // [pairs, I] f16 SwiGLU output, h * 2^-q
    float* h_scale;          // [pairs, I / 128] 2^q per 128-row segment
    float* partial;          // [pairs (pair id t*k + j), H]
    RouteBufs rb;
    WorkList wl;
    int* status;
    unsigned long long timeout_ns;
    int debug_stall;         // testing aid: the first routed expert never signals its gate/up items
    const RouteTable* rt;    // shared-memory routing table, or NULL (items come from wl)
};

// What changes between the expert phases of one launch (layer, counters, table).
struct ExpertLayer {
    int layer;
    int* queue;
    int* done;
    const RouteTable* rt;
};

// Item idx of the phase, from the routing table (rbu / rbd: row blocks of gate/up and down).
__device__ __forceinline__ ItemRec table_item(const RouteTable* rt, int idx, int rbu, int rbd) {
    const int n_gu = rt->n_chunks * rbu;
    const bool down = idx >= n_gu;
    const int j = down ? idx - n_gu : idx;
    const int nrb = down ? rbd : rbu;
    const int chunk = j / nrb, rbi = j % nrb;
    int lo = 0, hi = rt->n_active - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (rt->chunk0[mid] <= chunk) lo = mid; else hi = mid - 1;
    }
    const int tc = chunk - rt->chunk0[lo];
    ItemRec r;
    r.code = item_code(down ? 1 : 0, rbi, tc, lo);
    r.e = rt->e[lo];
    r.beg = rt->beg[lo] + tc * kTmaTok;
    r.ntok = min(kTmaTok, rt->cnt[lo] - tc * kTmaTok);
#pragma unroll
    for (int q = 0; q < kTmaTok; ++q) r.tok[q] = q < r.ntok ? (down ? rt->pair[r.beg + q] : rt->tok[r.beg + q]) : 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) r.pad[q] = 0;
    return r;
}

__device__ __forceinline__ ItemRec load_item(const ItemRec* src) {
    ItemRec r;
    const int4* s = reinterpret_cast<const int4*>(src);
    int4* d = reinterpret_cast<int4*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = __ldcg(s + i);
    return r;
}

struct SlotMeta {
    int kind, a, e, beg, ntok, stage, nstages, rb;
};

__device__ __forceinline__ float e8m0_f32(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}
// Byte k (0..3) of w as an E8M0 scale 2^(b-127): b << 23 for b >= 1; b = 0 gives
// 0x00400000 (the fp32 subnormal 2^-127) through the integer max.
__device__ __forceinline__ float e8m0_byte(uint32_t w, int k) {
    const uint32_t b = __byte_perm(w, 0u, 0x4440u + (uint32_t)k);
    return __uint_as_float(max(b << 23, 0x00400000u));
}

// Power of two 2^q with |v| * 2^-q in [2^14, 2^15) for the row maximum v (q = 0 for v = 0):
// keeps f16 values far from overflow while using its full precision.
__device__ __forceinline__ int f16_exponent_for(float amax) {
    if (!(amax > 0.0f)) return 0;
    const int q = ilogbf(amax) - 14;
    return q < -100 ? -100 : (q > 100 ? 100 : q);
}
__device__ __forceinline__ float exp2i(int q) {  // exact 2^q for -126 <= q <= 127
    return __uint_as_float((uint32_t)(q + 127) << 23);
}

// Waits on an mbarrier phase until it completes or the deadline passes (used to
// drain copies in flight before exiting; ignores the abort flag).
__device__ __forceinline__ bool drain_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() > deadline) return false;
    return true;
}

// Waits on an mbarrier phase, bounded by a deadline; returns false on timeout or abort.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline,
                                           const int* abort) {
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++spins & 255u) == 0) {
            if (globaltimer_ns() > deadline) return false;
            if (*reinterpret_cast<const volatile int*>(abort)) return false;
        }
    }
    return true;
}

// The same wait for a whole warp: every lane polls, and the warp leaves the loop
// together (completion seen by all lanes, or timeout / abort seen by any), so a
// warp never splits across a later __syncwarp.
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline,
                                                const int* abort) {
    uint32_t spins = 0;
    for (;;) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xFFFFFFFFu, done)) return true;
        if ((++spins & 255u) == 0) {
            const bool stop = globaltimer_ns() > deadline || *reinterpret_cast<const volatile int*>(abort) != 0;
            if (__any_sync(0xFFFFFFFFu, stop)) return false;
        }
    }
}

// Consumer work on one stage (the K half `kh`, 8 blocks of 32) for the 32 rows
// rbase..rbase+31 of the item, on the tensor cores.  Lane (g = lane/4, q = lane%4):
//   A: for MMA m (0, 1) of a block, rows g and g+8 of a 16-row tile, the code bytes
//      4q+2m, 4q+2m+1 of the block's 16 bytes -> block elements 8q+4m .. 8q+4m+3;
//   B: the same 4 elements of token g (one 16-byte load covers both MMAs).
// So the MMA pair of a block contracts exactly that block's 32 elements; its fp32
// tile (rows g, g+8; tokens 2q, 2q+1) is scaled by the rows' 2^(S-127) and added
// to acc[tile].  For down items the activations of every 128-element segment have
// their own power-of-two scale, applied once per segment (4 blocks).
template <int NT>
__device__ __forceinline__ void mma_stage(const uint8_t* slot, int rbase, int kh, int lane, float (&acc)[NT][4],
                                          bool seg_scaled) {
    const int g = lane >> 2, q = lane & 3;
    const uint8_t* box = slot + kh * (kTmaRows * 128);
    const uint8_t* act = slot + kSlotNib + kSlotScale + g * kActStride + kh * (kTmaKC / 2) * 2 + 16 * q;
    // scale bytes of this K half: rows rbase + 16 tt + g (+8)
    uint2 sc[NT][2];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8)
            sc[tt][h8] = *reinterpret_cast<const uint2*>(slot + kSlotNib + (rbase + 16 * tt + 8 * h8 + g) * 16 + kh * 8);
    float segf[2][2] = {{1.0f, 1.0f}, {1.0f, 1.0f}};   // [segment][token 2q, 2q+1]
    if (seg_scaled) {
        const float* aux = reinterpret_cast<const float*>(slot + kSlotNib + kSlotScale + kSlotAct);
#pragma unroll
        for (int sg = 0; sg < 2; ++sg) {
            segf[sg][0] = aux[(2 * q) * 4 + 2 * kh + sg];
            segf[sg][1] = aux[(2 * q + 1) * 4 + 2 * kh + sg];
        }
    }
#pragma unroll
    for (int sg = 0; sg < 2; ++sg) {
        float part[NT][4];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[tt][i] = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = sg * 4 + jj;
            const uint4 xv = *reinterpret_cast<const uint4*>(act + j * 64);
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const int r0 = rbase + 16 * tt + g;   // r0 & 7 == (r0 + 8) & 7 == g
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(box + r0 * 128 + ((j ^ g) << 4) + 4 * q);
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(box + (r0 + 8) * 128 + ((j ^ g) << 4) + 4 * q);
                uint32_t c0[4], c1[4];   // bytes 0..3 of rows g and g+8
                e2m1x8_to_f16x2(w0, c0);
                e2m1x8_to_f16x2(w1, c1);
                const uint32_t a0[4] = {c0[0], c1[0], c0[1], c1[1]};
                const uint32_t a1[4] = {c0[2], c1[2], c0[3], c1[3]};
                const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float d[4];
                mma_16816_f16(d, a0, xv.x, xv.y, zero);
                mma_16816_f16(d, a1, xv.z, xv.w, d);
                const float s0 = e8m0_byte(j < 4 ? sc[tt][0].x : sc[tt][0].y, j & 3);
                const float s1 = e8m0_byte(j < 4 ? sc[tt][1].x : sc[tt][1].y, j & 3);
                part[tt][0] = fmaf(d[0], s0, part[tt][0]);
                part[tt][1] = fmaf(d[1], s0, part[tt][1]);
                part[tt][2] = fmaf(d[2], s1, part[tt][2]);
                part[tt][3] = fmaf(d[3], s1, part[tt][3]);
            }
        }
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            acc[tt][0] = fmaf(part[tt][0], segf[sg][0], acc[tt][0]);
            acc[tt][1] = fmaf(part[tt][1], segf[sg][1], acc[tt][1]);
            acc[tt][2] = fmaf(part[tt][2], segf[sg][0], acc[tt][2]);
            acc[tt][3] = fmaf(part[tt][3], segf[sg][1], acc[tt][3]);
        }
    }
}

// Shared memory of the expert phase: the slot ring, the K-half exchange area,
// the ring / epilogue mbarriers and the per-slot metadata.
struct ExpertSmem {
    uint8_t* slots;
    float* epi;          // [2][128 rows][8 tokens]
    uint64_t* full;      // [kTmaStages]
    uint64_t* empty;     // [kTmaStages]
    uint64_t* epi_bar;
    SlotMeta* meta;      // [kTmaStages]
    RouteTable* rt;      // small-block routing table (persistent forward)
};

__device__ __forceinline__ ExpertSmem expert_smem(uint8_t* smem_raw) {
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    ExpertSmem sm;
    sm.slots = smem;
    sm.epi = reinterpret_cast<float*>(smem + kTmaStages * kSlotBytes);
    sm.full = reinterpret_cast<uint64_t*>(smem + kTmaStages * kSlotBytes + kEpiBytes);
    sm.empty = sm.full + kTmaStages;
    sm.epi_bar = sm.empty + kTmaStages;
    sm.meta = reinterpret_cast<SlotMeta*>(sm.epi_bar + 1);
    sm.rt = reinterpret_cast<RouteTable*>(sm.meta + kTmaStages);
    return sm;
}

// One thread initialises the barriers (then the block synchronises).
__device__ __forceinline__ void expert_smem_init(const ExpertSmem& sm) {
    for (int s = 0; s < kTmaStages; ++s) {
        mbar_init(&sm.full[s], 1);
        mbar_init(&sm.empty[s], kTmaConsumerWarps);
    }
    mbar_init(sm.epi_bar, kTmaConsumerWarps);
    fence_barrier_init();
}

// Producer of one expert phase (one thread): claims items until the queue is
// empty, streams their stages into the ring and finally publishes an END slot.
// `it` is the ring position, carried across phases.  Returns false on a timeout.
__device__ bool expert_produce(const TmaMaps& maps, const ExpertArgs& args, const ExpertLayer lay, const ExpertSmem& sm,
                               uint32_t& it, unsigned long long deadline) {
    uint8_t* slots = sm.slots;
    uint64_t* full = sm.full;
    uint64_t* empty = sm.empty;
    SlotMeta* meta = sm.meta;
    const int H = args.H, I = args.I;
    {
        {
            // work-list data is written by another CTA in the same launch: read it from L2
            const int rbu = I / kTmaRows, rbd = H / kTmaRows;
            const int n_items = lay.rt ? lay.rt->n_chunks * (rbu + rbd) : __ldcg(args.wl.n_items);
            bool finished = false, failed = false;
            // one item of lookahead: the next record is claimed and loaded while
            // the current item's stages are issued
            int next_idx = atomicAdd(lay.queue, 1);
            ItemRec next{};
            if (next_idx < n_items)
                next = lay.rt ? table_item(lay.rt, next_idx, rbu, rbd) : load_item(args.wl.items + next_idx);
            while (!finished && !failed) {
                const int idx = next_idx;
                const ItemRec cur = next;
                const bool end = idx >= n_items;
                if (!end) {
                    next_idx = atomicAdd(lay.queue, 1);
                    if (next_idx < n_items)
                        next = lay.rt ? table_item(lay.rt, next_idx, rbu, rbd) : load_item(args.wl.items + next_idx);
                }
                int kind = 0, a = 0, e = 0, beg = 0, ntok = 0, nstages = 1, rb = 0;
                if (!end) {
                    kind = (cur.code >> 30) & 1;
                    rb = (cur.code >> 20) & 0x3FF;
                    a = cur.code & 0x7FF;
                    e = cur.e;
                    beg = cur.beg;
                    ntok = cur.ntok;
                    nstages = kind == kItemGateUp ? 2 * (H / kTmaKC) : I / kTmaKC;
                }
                bool h_ready = kind == kItemGateUp;
                for (int s = 0; s < nstages; ++s) {
                    const int slot = it % kTmaStages;
                    const uint32_t n = it / kTmaStages;
                    if (!wait_phase(&empty[slot], (n & 1) ^ 1, deadline, args.wl.abort)) { failed = true; break; }
                    SlotMeta m;
                    m.kind = end ? -1 : kind; m.a = a; m.e = e; m.beg = beg; m.ntok = ntok;
                    m.stage = s; m.nstages = nstages; m.rb = rb;
                    meta[slot] = m;
                    if (end) { mbar_arrive(&full[slot]); ++it; finished = true; break; }
                    uint8_t* dst = slots + slot * kSlotBytes;
                    const uint32_t bytes = kSlotNib + kSlotScale + (uint32_t)ntok * (kTmaKC * 2 + 16u);
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    ++it;   // this slot now has copies in flight
                    const CUtensorMap* mq;
                    const CUtensorMap* ms;
                    int k0, row0;
                    if (kind == kItemGateUp) {
                        mq = (s & 1) ? &maps.up_q : &maps.gate_q;
                        ms = (s & 1) ? &maps.up_s : &maps.gate_s;
                        k0 = (s >> 1) * kTmaKC;
                        row0 = e * I + rb * kTmaRows;
                    } else {
                        mq = &maps.down_q;
                        ms = &maps.down_s;
                        k0 = s * kTmaKC;
                        row0 = e * H + rb * kTmaRows;
                    }
                    tma_load_2d(dst, mq, k0 / 2, row0, &full[slot]);
                    tma_load_2d(dst + kTmaRows * 128, mq, k0 / 2 + 128, row0, &full[slot]);
                    tma_load_2d(dst + kSlotNib, ms, k0 / 32, row0, &full[slot]);
                    // L2 prefetch of this item's matrix two stages ahead
                    if (s + 2 < nstages) {
                        const int s2 = s + 2;
                        const CUtensorMap* mq2 = kind == kItemGateUp ? ((s2 & 1) ? &maps.up_q : &maps.gate_q) : mq;
                        const int k2 = kind == kItemGateUp ? (s2 >> 1) * kTmaKC : s2 * kTmaKC;
                        tma_prefetch_2d(mq2, k2 / 2, row0);
                        tma_prefetch_2d(mq2, k2 / 2 + 128, row0);
                    }
                    uint8_t* act_dst = dst + kSlotNib + kSlotScale;
                    if (kind == kItemGateUp) {
                        uint8_t* aux = act_dst + kSlotAct;
                        for (int i = 0; i < ntok; ++i) {
                            bulk_load(act_dst + i * kActStride, args.act16 + (size_t)cur.tok[i] * H + k0,
                                      kTmaKC * 2, &full[slot]);
                            // the 4 segment factors (128 activations each) of this stage's K range
                            bulk_load(aux + i * 16, args.act_fac + (size_t)cur.tok[i] * (H / 128) + k0 / 128, 16,
                                      &full[slot]);
                        }
                    } else {
                        if (!h_ready) {
                            // every gate/up item of this expert must have stored h
                            const int need = lay.rt ? (lay.rt->cnt[a] + kTmaTok - 1) / kTmaTok * rbu
                                                     : __ldcg(args.wl.need + a);
                            uint32_t spins = 0;
                            while (ld_acquire_gpu(lay.done + a) < need) {
                                if ((++spins & 63u) == 0 &&
                                    (globaltimer_ns() > deadline ||
                                     *reinterpret_cast<const volatile int*>(args.wl.abort))) {
                                    failed = true;
                                    break;
                                }
                            }
                            fence_proxy_async_global();
                            h_ready = true;
                        }
                        // issued even after a failed wait, so that the armed stage completes
                        uint8_t* aux = act_dst + kSlotAct;
                        for (int i = 0; i < ntok; ++i) {
                            bulk_load(act_dst + i * kActStride, args.h16 + (size_t)(beg + i) * I + k0, kTmaKC * 2,
                                      &full[slot]);
                            // the 4 segment scales (128 h values each) of this stage's K range
                            bulk_load(aux + i * 16, args.h_scale + (size_t)(beg + i) * (I / 128) + k0 / 128, 16,
                                      &full[slot]);
                        }
                        if (failed) break;
                    }
                }
            }
            if (failed) {
                if (atomicExch(args.wl.abort, 1) == 0) raise_status(args.status, MOE_ERR_TIMEOUT, lay.layer * 65536);
                // every copy this CTA issued must land before the CTA exits
                const uint32_t issued = it < (uint32_t)kTmaStages ? it : (uint32_t)kTmaStages;
                for (uint32_t q = 0; q < issued; ++q) {
                    const uint32_t last = it - 1 - q;
                    drain_phase(&full[last % kTmaStages], (last / kTmaStages) & 1,
                                globaltimer_ns() + args.timeout_ns);
                }
            }
            return !failed;
        }
    }
}

// Consumers of one expert phase (warps 0..kTmaConsumerWarps-1): consume slots until
// the END slot (which they release too).  `it` and `epi_uses` are carried across
// phases.  Returns false on a timeout / abort.
__device__ bool expert_consume(const ExpertArgs& args, const ExpertLayer lay, const ExpertSmem& sm, uint32_t& it,
                               uint32_t& epi_uses, int warp, int lane, unsigned long long deadline) {
    const uint8_t* slots = sm.slots;
    float* epi = sm.epi;
    uint64_t* full = sm.full;
    uint64_t* empty = sm.empty;
    uint64_t* epi_bar = sm.epi_bar;
    const SlotMeta* meta = sm.meta;
    const int H = args.H, I = args.I;
    const int rp = warp % kTmaRowGroups, kh = warp / kTmaRowGroups;
    const int rbase = 16 * kTmaTiles * rp;
    const int g = lane >> 2, q = lane & 3;
    float accG[kTmaTiles][4], accU[kTmaTiles][4];
#pragma unroll
    for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
        for (int i = 0; i < 4; ++i) accG[tt][i] = accU[tt][i] = 0.0f;
    // consumer-wide barrier on an mbarrier (8 warp arrivals) with a bounded wait
    auto consumer_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_bar);
        const bool ok = warp_wait_phase(epi_bar, epi_uses & 1, deadline, args.wl.abort);
        ++epi_uses;
        return ok;
    };
    // this thread's outputs: rows rbase + 16 tt + g + 8 h8, tokens 2q + c, value index 2 h8 + c
    auto row_of = [&](int tt, int i) { return rbase + 16 * tt + g + 8 * (i >> 1); };
    auto tok_of = [&](int i) { return 2 * q + (i & 1); };
    bool failed = false;
    for (;; ++it) {
        const int slot = it % kTmaStages;
        const uint32_t n = it / kTmaStages;
        if (!warp_wait_phase(&full[slot], n & 1, deadline, args.wl.abort)) { failed = true; break; }
        const SlotMeta m = meta[slot];
        if (m.kind < 0) {   // END: release the slot so the ring stays in step for the next phase
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++it;
            break;
        }
        const uint8_t* sl = slots + slot * kSlotBytes;
        if (m.stage == 0) {
#pragma unroll
            for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) accG[tt][i] = accU[tt][i] = 0.0f;
        }
        // scale bytes 0xFF (NaN) are invalid input: check this thread's share of the tile
        {
            const int rr = (warp * 32 + lane) * 16 / kTmaConsumerWarps;   // 16 B of scales per 256/NW threads
            const uint2 sc = kTmaConsumerWarps == 8
                                 ? *reinterpret_cast<const uint2*>(sl + kSlotNib + (warp * 16 + (lane >> 1)) * 16 +
                                                                   (lane & 1) * 8)
                                 : make_uint2(*reinterpret_cast<const uint32_t*>(sl + kSlotNib + rr * 4), 0u);
            const uint32_t ff = (sc.x & (sc.x >> 1) & (sc.x >> 2) & (sc.x >> 3) & (sc.x >> 4) & (sc.x >> 5) &
                                 (sc.x >> 6) & (sc.x >> 7) & 0x01010101u) |
                                (sc.y & (sc.y >> 1) & (sc.y >> 2) & (sc.y >> 3) & (sc.y >> 4) & (sc.y >> 5) &
                                 (sc.y >> 6) & (sc.y >> 7) & 0x01010101u);
            if (ff) raise_status(args.status, MOE_ERR_BAD_SCALE, lay.layer * 65536 + m.e);
        }
        if (m.kind == kItemGateUp) {
            if (m.stage & 1) mma_stage<kTmaTiles>(sl, rbase, kh, lane, accU, true);
            else mma_stage<kTmaTiles>(sl, rbase, kh, lane, accG, true);
        } else {
            mma_stage<kTmaTiles>(sl, rbase, kh, lane, accG, true);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        if (m.stage != m.nstages - 1) continue;
        // ---- epilogue: the K-half-1 warps hand their sums to the K-half-0 warps
        // through shared memory (epi[row][token], gate then up), which finish.
        float* exG = epi;                        // [128 rows][8 tokens]
        float* exU = epi + kTmaRows * kTmaTok;
        if (kh == 1) {
#pragma unroll
            for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    exG[row_of(tt, i) * kTmaTok + tok_of(i)] = accG[tt][i];
                    exU[row_of(tt, i) * kTmaTok + tok_of(i)] = accU[tt][i];
                }
        }
        if (!consumer_sync()) { failed = true; break; }
        if (m.kind == kItemGateUp) {
            float hv[kTmaTiles][4];
            float mx0 = 0.0f, mx1 = 0.0f;   // tokens 2q, 2q+1 over this thread's rows
            if (kh == 0) {
#pragma unroll
                for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = row_of(tt, i), c = tok_of(i);
                        const float gg = accG[tt][i] + exG[r * kTmaTok + c];
                        const float uu = accU[tt][i] + exU[r * kTmaTok + c];
                        const float h = silu(gg) * uu;
                        hv[tt][i] = h;
                        if (i & 1) mx1 = fmaxf(mx1, fabsf(h)); else mx0 = fmaxf(mx0, fabsf(h));
                    }
            }
            if (!consumer_sync()) { failed = true; break; }   // ex reads done: reuse epi for maxima
            // reduce over the 8 lanes that share q (same tokens), then over the 4 row groups
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
            }
            if (kh == 0 && g == 0) {
                epi[rp * kTmaTok + 2 * q] = mx0;
                epi[rp * kTmaTok + 2 * q + 1] = mx1;
            }
            if (!consumer_sync()) { failed = true; break; }
            if (kh == 0) {
                const int segs = I / 128;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int tok = 2 * q + c;
                    if (tok < m.ntok) {
                        float mx = 0.0f;
#pragma unroll
                        for (int r8 = 0; r8 < kTmaRowGroups; ++r8) mx = fmaxf(mx, epi[r8 * kTmaTok + tok]);
                        const int qe = f16_exponent_for(mx);
                        const float inv = exp2i(-qe);
                        const size_t pos = (size_t)(m.beg + tok);
#pragma unroll
                        for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
                            for (int h8 = 0; h8 < 2; ++h8)
                                args.h16[pos * I + m.rb * kTmaRows + row_of(tt, 2 * h8)] =
                                    __float2half_rn(hv[tt][2 * h8 + c] * inv);
                        if (rp == 0 && g == 0) args.h_scale[pos * segs + m.rb] = exp2i(qe);
                    }
                }
            }
            if (!consumer_sync()) { failed = true; break; }
            if (threadIdx.x == 0 && !(args.debug_stall && m.a == 0)) {
                __threadfence();
                fence_proxy_async_global();
                red_release_add_gpu(lay.done + m.a, 1);
            }
        } else {
            if (kh == 0) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int tok = 2 * q + c;
                    if (tok < m.ntok) {
                        const int pair = lay.rt ? lay.rt->pair[m.beg + tok] : __ldcg(args.rb.perm + m.beg + tok);
#pragma unroll
                        for (int tt = 0; tt < kTmaTiles; ++tt)
#pragma unroll
                            for (int h8 = 0; h8 < 2; ++h8) {
                                const int r = row_of(tt, 2 * h8);
                                args.partial[(size_t)pair * H + m.rb * kTmaRows + r] =
                                    accG[tt][2 * h8 + c] + exG[r * kTmaTok + tok];
                            }
                    }
                }
            }
            if (!consumer_sync()) { failed = true; break; }
        }
    }
    if (failed && lane == 0) {
        if (atomicExch(args.wl.abort, 1) == 0) raise_status(args.status, MOE_ERR_TIMEOUT, lay.layer * 65536);
    }
    return !failed;
}

__global__ void __launch_bounds__(kTmaThreads, 1) expert_tma_kernel(const __grid_constant__ TmaMaps maps,
                                                                    const ExpertArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const ExpertSmem sm = expert_smem(smem_raw);
    if (threadIdx.x == 0) expert_smem_init(sm);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned long long deadline = globaltimer_ns() + args.timeout_ns;
    uint32_t it = 0, epi_uses = 0;
    const ExpertLayer lay{args.layer, args.wl.queue, args.wl.done, args.rt};
    if (warp == kTmaConsumerWarps) {
        if (lane == 0) {
            prefetch_tensormap(&maps.gate_q);
            prefetch_tensormap(&maps.up_q);
            prefetch_tensormap(&maps.down_q);
            prefetch_tensormap(&maps.gate_s);
            prefetch_tensormap(&maps.up_s);
            prefetch_tensormap(&maps.down_s);
            expert_produce(maps, args, lay, sm, it, deadline);
        }
        return;
    }
    expert_consume(args, lay, sm, it, epi_uses, warp, lane, deadline);
}

// Builds the work list of one layer from the grouping: for every routed expert
// (active index a) and every chunk of up to 8 of its tokens, I/128 gate/up
// items, then H/128 down items, each with its full record.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) build_items_kernel(RouteBufs rb, int H, int I, int k, WorkList wl, int T) {
    __shared__ int s_gu[kMaxExperts + 1];
    __shared__ int s_act[kMaxExperts], s_beg[kMaxExperts], s_cnt[kMaxExperts];
    __shared__ int s_scan[64];
    extern __shared__ int s_perm[];   // [T * k] pair id of each perm position
    const int n_active = rb.active[0];
    const int rbu = I / kTmaRows, rbd = H / kTmaRows;
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
    if (a < n_active) {
        s_gu[a] = off;
        wl.need[a] = chunks * rbu;
        wl.done[a] = 0;
    }
    __syncthreads();
    const int n_gu = total_chunks * rbu;
    if (threadIdx.x == 0) {
        wl.n_items[0] = n_gu + total_chunks * rbd;
        wl.n_items[1] = n_gu;
        *wl.queue = 0;
        *wl.abort = 0;
    }
    // item i -> (kind, chunk, row block); chunk -> (active expert aa, token chunk tc)
    // by a binary search of the chunk prefix.  Gate/up items first, then down items.
    const int total = total_chunks * (rbu + rbd);
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const bool down = i >= n_gu;
        const int j = down ? i - n_gu : i;
        const int nrb = down ? rbd : rbu;
        const int chunk = j / nrb, rbi = j % nrb;
        int lo = 0, hi = n_active - 1;          // last aa with s_gu[aa] <= chunk
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_gu[mid] <= chunk) lo = mid; else hi = mid - 1;
        }
        const int aa = lo, tc = chunk - s_gu[aa];
        ItemRec r;
        r.code = item_code(down ? kItemDown : kItemGateUp, rbi, tc, aa);
        r.e = s_act[aa];
        r.beg = s_beg[aa] + tc * kTmaTok;
        r.ntok = min(kTmaTok, s_cnt[aa] - tc * kTmaTok);
#pragma unroll
        for (int q = 0; q < kTmaTok; ++q) r.tok[q] = q < r.ntok ? (down ? s_perm[r.beg + q] : s_perm[r.beg + q] / k) : 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) r.pad[q] = 0;
        wl.items[i] = r;
    }
}

// Input staging of one layer, one block of 1024 threads per token:
//   norm_w == NULL: act[t] = fp32(x[t]) (x bf16), and resid[t] = act[t] when resid != NULL;
//   norm_w != NULL: act[t] = resid[t] * w / sqrt(mean(resid[t]^2) + eps)  (RMSNorm);
// then act16[t] = f16(act[t] * 2^-p_t) with 2^p_t from the row maximum (exact for
// bf16-valued rows), and 2^p_t as the factor of every 128-wide segment of the row.
constexpr int kPrepThreads = 1024;
__global__ void __launch_bounds__(kPrepThreads) prep_layer_kernel(const __nv_bfloat16* __restrict__ x, int H,
                                                                  float* resid, const __nv_bfloat16* __restrict__ norm_w,
                                                                  float eps, float* __restrict__ act,
                                                                  __half* __restrict__ act16,
                                                                  float* __restrict__ act_fac) {
    __shared__ float red[2][32];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kPer = 16;   // H <= 16384: at most 16 values per thread
    float v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int h = threadIdx.x + i * kPrepThreads;
        v[i] = 0.0f;
        if (h < H) v[i] = norm_w ? resid[(size_t)t * H + h] : __bfloat162float(x[(size_t)t * H + h]);
    }
    if (norm_w) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) red[0][warp] = ss;
        __syncthreads();
        float tot = 0.0f;
        for (int i = 0; i < 32; ++i) tot += red[0][i];
        const float inv = 1.0f / sqrtf(tot / (float)H + eps);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int h = threadIdx.x + i * kPrepThreads;
            if (h < H) v[i] = v[i] * inv * __bfloat162float(norm_w[h]);
        }
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[1][warp] = m;
    __syncthreads();
    float mx = 0.0f;
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, red[1][i]);
    const int p = f16_exponent_for(mx);
    const float inv = exp2i(-p);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int h = threadIdx.x + i * kPrepThreads;
        if (h < H) {
            act[(size_t)t * H + h] = v[i];
            act16[(size_t)t * H + h] = __float2half_rn(v[i] * inv);
            if (resid && !norm_w) resid[(size_t)t * H + h] = v[i];
        }
    }
    for (int i = threadIdx.x; i < H / 128; i += blockDim.x) act_fac[(size_t)t * (H / 128) + i] = exp2i(p);
}

}  // namespace moe
