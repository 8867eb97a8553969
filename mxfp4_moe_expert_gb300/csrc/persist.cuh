// Persistent forward: one cooperative launch runs every phase of every layer
// ("MiMo 把 1T 模型推到每秒千 token", persistent engine kernel section: the whole
// pipeline stays resident instead of one launch per operator; implementation
// guide "关键实现细节" item 3: per-launch gaps of 5-10 us and 10-30% operator-boundary
// overhead at high token rates).  One CTA per SM, the expert kernel's block
// shape (16 warps) and tensor-memory allocation.  Per layer of a plain input x:
//   [router]           one block of <= 8 tokens: CTA b computes whole logit rows of a
//                      few experts from x and their weight rows in shared memory;
//                      larger blocks: units of (32 experts x 256..1024 columns x a token
//                      block), partial logits summed by the whole grid after the
//                      barrier; every warp of the grid: x as the experts' operand (8
//                      E2M1 terms per MX block)
//   -- grid barrier --
//   [route]            small blocks (T*k <= 64): every CTA takes the top-k and groups
//                      the pairs in its own shared memory (identical results
//                      everywhere; CTA 0 publishes them after its expert phase);
//                      larger blocks: top-k on every warp, the grouping by CTA 0 while
//                      the other CTAs wait on a release flag, then every CTA builds its
//                      share of the work list and gathers the operand per chunk
//                      (chunks of 32 pairs x 4 terms, all 128 rows of the MMA)
//   [experts]          the work-queue expert phase of expert_tc.cuh (TcSmall or TcWide)
//   -- grid barrier --
//   [combine]          all CTAs: gate-weighted sum of the pair outputs (grid-stride
//                      over (token, 4 columns))
// A residual stack has no router phase: its combine units (token, 256 columns) add the
// residual, keep the block sums of squares and form the next layer's router products and
// operand from r * w_norm (prep_unit); the routing scales the logits and the gate/up
// epilogue scales g and u by 1 / rms (one factor per token).  Per layer: [route]
// [experts] -- barrier -- [combine + next layer's inputs] -- barrier --.
// The counters and the barrier word in the workspace are at rest between launches (see
// persist_kernel).  Every wait is bounded by the forward's deadline; a timeout sets the
// status word and the abort flag, and every CTA leaves at its next wait.
#pragma once

#include "expert_tc.cuh"
#include "route.cuh"

namespace moe {

constexpr int kMaxPersistLayers = 8;
constexpr int kPRouteExperts = 32;   // 16 warps x 2 expert rows
constexpr int kPRouteSlice = 1024;   // columns per router unit: 4 sub-chunks of 256 (8 per lane)
constexpr int kPRouteSub = 256;
constexpr int kPRouteTok = 8;        // tokens per round
constexpr int kCombineChunk = 256;   // columns per combine unit (and per sum-of-squares block)

struct PersistLayer {
    TcMaps maps;
    const __nv_bfloat16* router_w;
    const float* router_b;
    const __nv_bfloat16* norm_w;
};

struct PersistDebug {    // device pointers, [L, ...] each, or NULL
    int* idx;
    float* gate;
    int* counts;
    int* offsets;
    int* perm;
};

struct PersistParams {
    PersistLayer layer[kMaxPersistLayers];
    int L, T, H, I, E, k;
    int e_begin, e_end;
    int y_bf16;
    int norm;          // pre-norm residual stack
    int init_from_x;   // the residual starts from x (first launch of a stack)
    int write_y;       // the last layer of this launch writes y
    int layer_base;    // index of layer[0] in the whole stack
    float eps;
    const __nv_bfloat16* x;
    void* y;
    float* resid;      // [T, H] (stack)
    uint8_t* xb4;      // expert operand of the layer input (expert_tc.cuh layouts)
    uint8_t* xsf;
    float* ss;         // [T, H / 256] sums of squares of the residual per column block
    float* rpart;      // [H / rslice, T, E] router slice partials
    int rslice;        // columns per router unit (256, 512 or 1024; divides H)
    int rfull;         // experts per whole-row router unit (router_full_unit), or 0: column-sliced units
    int chunk;         // pairs per chunk of a block routed through the workspace (32 dense, or 16)
    int terms;         // E2M1 terms per activation in those chunks (4 dense, or 8): 128 operand rows
    int rtok;          // tokens per router unit (T for blocks routed in shared memory; else a multiple of 8 G)
    int* rcnt;         // [kMaxPersistLayers, 32] finished router units per expert group (0 at rest)
    unsigned long long* tstamp;   // CTA 0's %globaltimer at phase ends (or NULL)
    TcArgs ta;         // expert phase: operands, partial, status, timeout (per-layer fields set per layer)
    RouteBufs rb;
    WorkList wl;       // items / n_items / abort for larger blocks
    int* queues;       // [kMaxPersistLayers] expert-phase queue per layer (0 at rest)
    int* dones;        // [kMaxPersistLayers, chunk_stride] finished gate/up items per chunk (0 at rest)
    int chunk_stride;
    unsigned* bar;     // grid barrier word (low 31 bits 0 at rest; see grid_arrive)
    int* route_flag;   // layers routed so far in this launch (0 at rest)
    const unsigned long long* state_tag;   // the workspace's state tag (see persist_kernel)
    unsigned long long tag;                // its expected value
    float* tscale;     // [T] per-token 1 / rms of a residual stack (blocks routed through the workspace)
    PersistDebug dbg;
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool aborted(const int* abort) {
    return *reinterpret_cast<const volatile int*>(abort) != 0;
}

// All CTAs of the grid meet; bounded.  grid_arrive announces this CTA (after every
// thread's earlier writes), grid_wait waits for every CTA's arrival at the same barrier;
// work between the two must not depend on the other CTAs.  grid_wait returns false (in
// every thread) on timeout / abort.
// One 32-bit word serves every barrier of every launch and returns to its resting value
// by itself: each CTA adds 1, except CTA 0, which adds 2^31 - (G - 1).  The G additions
// of one barrier sum to 2^31, so the low 31 bits are back to 0 and bit 31 has flipped;
// bit 31 flips only with the last addition (before it, the sum is short of 2^31 or CTA
// 0's term has borrowed from bit 31), and each CTA waits until bit 31 differs from the
// value its own addition returned.  No launch needs the word cleared.
__device__ __forceinline__ void grid_arrive(unsigned* bar, unsigned& token, bool withhold = false) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
        token = withhold ? ld_acquire_u32(bar) : atomicAdd(bar, add);
    }
}
__device__ __forceinline__ bool grid_wait(unsigned* bar, unsigned token, unsigned long long deadline, int* abort,
                                          int* status) {
    int failed = 0;
    if (threadIdx.x == 0) {
        uint32_t spins = 0;
        while (((ld_acquire_u32(bar) ^ token) & 0x80000000u) == 0u) {
            if ((++spins & 63u) == 0 && (globaltimer_ns() > deadline || aborted(abort))) {
                failed = 1;
                if (atomicExch(abort, 1) == 0) raise_status(status, MOE_ERR_TIMEOUT, -1);
                break;
            }
        }
    }
    return __syncthreads_or(failed) == 0;
}
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned& token, unsigned long long deadline,
                                          int* abort, int* status, bool withhold = false) {
    grid_arrive(bar, token, withhold);
    return grid_wait(bar, token, deadline, abort, status);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

__device__ __forceinline__ float block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < nw; ++i) t = fmaxf(t, red[i]);
    return t;
}

// Exclusive scan by one warp of n <= 1024 ints (lane l owns a contiguous run).
// Returns the total to every lane.
__device__ __forceinline__ int warp_excl_scan(int* v, int n) {
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int b = min(n, lane * per), e = min(n, b + per);
    int s = 0;
    for (int i = b; i < e; ++i) s += v[i];
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    int run = incl - s;
    for (int i = b; i < e; ++i) {
        const int c = v[i];
        v[i] = run;
        run += c;
    }
    return __shfl_sync(0xFFFFFFFFu, incl, 31);
}

// 1/sqrt(mean(r^2) + eps) of token t from the block sums of squares (summed in
// block order by one warp: every caller gets the same value).
__device__ __forceinline__ float inv_rms(const PersistParams& p, int t) {
    const int lane = threadIdx.x & 31;
    const int nc = p.H / kCombineChunk;   // <= 64
    const float v0 = lane < nc ? __ldcg(p.ss + (size_t)t * nc + lane) : 0.0f;
    const float v1 = lane + 32 < nc ? __ldcg(p.ss + (size_t)t * nc + lane + 32) : 0.0f;
    float tot = 0.0f;
    for (int c = 0; c < nc; ++c) tot += c < 32 ? __shfl_sync(0xFFFFFFFFu, v0, c) : __shfl_sync(0xFFFFFFFFu, v1, c - 32);
    return 1.0f / sqrtf(tot / (float)p.H + p.eps);
}

// The block is routed by every CTA in its own shared memory (route_small) rather than
// through the workspace (topk_tokens / route_phase / build_items_slice).
__device__ __forceinline__ bool route_is_small(const PersistParams& p) {
    return p.T * p.k <= kRtMaxPairs && p.T * p.E <= 8192;
}

// Router units (a plain input x; a residual stack forms its router products in prep_unit)
// process G groups of 8 tokens per pass: G = 1 for a single 8-token block (the 16 warps
// split K); larger blocks G = 4 (1024-column slices) or 8 (narrower).
__device__ __forceinline__ int router_groups(const PersistParams& p) {
    if (p.T <= kPRouteTok) return 1;
    return 4 * (p.rslice >= 1024 ? 1 : 2);
}
// Shared-memory layout of a router unit (slot area): the staged input rows
// [8 G rows][stride] at 0, the weight rows [32][stride] at router_wbase.  stride =
// rslice * 2 + 16 bytes (rows padded by 16 bytes: conflict-free ldmatrix).  The warps'
// sums [16][32][24] floats (48 KB) reuse offset 0 after the MMAs.
__device__ __forceinline__ uint32_t router_stride(const PersistParams& p) { return (uint32_t)p.rslice * 2 + 16; }
// Router units: (weight slice r = (expert group eg of 32, column slice sl), token block tb),
// u = r * token blocks + tb with r = eg * slices + sl: the token blocks of one weight
// slice are adjacent.
__device__ __forceinline__ int router_egroups(const PersistParams& p) { return (p.E + kPRouteExperts - 1) / kPRouteExperts; }
__device__ __forceinline__ int router_tblocks(const PersistParams& p) { return (p.T + p.rtok - 1) / p.rtok; }
__device__ __forceinline__ int router_units(const PersistParams& p) {
    return router_egroups(p) * (p.H / p.rslice) * router_tblocks(p);
}
// This CTA's router units, first / end / step: blocks routed in shared memory take units
// b, b + grid, ... (one token block each); larger blocks (kContiguous) a contiguous range,
// so that consecutive units of a CTA mostly share their weight slice (kept in shared memory).
template <bool kContiguous>
__device__ __forceinline__ int router_first(int units) {
    return kContiguous ? (int)((long long)units * blockIdx.x / gridDim.x) : (int)blockIdx.x;
}
template <bool kContiguous>
__device__ __forceinline__ int router_end(int units) {
    return kContiguous ? (int)((long long)units * (blockIdx.x + 1) / gridDim.x) : units;
}
template <bool kContiguous>
__device__ __forceinline__ int router_step() { return kContiguous ? 1 : (int)gridDim.x; }
__device__ __forceinline__ uint32_t router_wbase(const PersistParams& p) {
    const uint32_t a = max(8u * router_groups(p) * router_stride(p), 16u * 768u * 4u);
    return (a + 1023u) & ~1023u;
}

// Router-weight copies: the weight rows of one router unit (up to 32 experts x rslice
// columns, bf16) into shared memory (router_wbase into the slot area, rows padded), as
// 16-byte cp.async copies spread over every thread of the CTA (L2 evict-first): all in
// flight at once, without a copy-engine request per row.  They have landed once every
// thread has passed cp.async.wait_all and the block has synchronised.  State in shared
// memory (rstate): [2] / [3] unit / layer whose copies were issued ahead of time (-1:
// none), [5] / [6] weight slice / layer in shared memory (-1: none), [8] router_unit's
// decision to fetch.
__device__ __forceinline__ void router_fetch(const PersistParams& p, const PersistLayer& ly, int u,
                                             const TcSmem& sm) {   // whole CTA
    const int n_sl = p.H / p.rslice;
    const int r = u / router_tblocks(p);   // the token block does not change the weights
    const int eg = r / n_sl, sl = r % n_sl;
    const int ne = min(kPRouteExperts, p.E - eg * kPRouteExperts);
    const int n16 = p.rslice / 8;          // 16-byte pieces per row
    const uint32_t stride = router_stride(p), dst = smem_u32(sm.slots + router_wbase(p));
    const uint64_t pol = l2_evict_first_policy();
    const __nv_bfloat16* src = ly.router_w + (size_t)eg * kPRouteExperts * p.H + (size_t)sl * p.rslice;
    for (int i = threadIdx.x; i < ne * n16; i += blockDim.x) {
        const int row = i / n16, c = (i % n16) * 8;
        cp_async_16_hint(dst + (uint32_t)row * stride + (uint32_t)c * 2, src + (size_t)row * p.H + c, pol);
    }
}

// Router unit u = (token block of p.rtok tokens, expert group g of 32, column slice s of
// p.rslice columns): partial logits of the group over the slice for the block's tokens,
// 8 G tokens per pass, on the tensor cores: per 8-token group D [32 experts x 8 tokens] =
// W [32 x K] . X^T with the bf16 input x as it is (fp32 accumulation; every bf16 x bf16
// product is exact), copied into shared memory by cp.async.  The 16 / G warps of a group
// split K; their results are summed in a fixed order.  The weight rows come into shared
// memory by router_fetch (issued ahead of time where possible).  The unit that finishes a
// group last (a counter per group) sums the group's slice partials in slice order and
// writes its logits (+ bias): the result does not depend on which unit comes last.
__device__ __noinline__ void router_unit(const PersistParams& p, const PersistLayer& ly, int l, int u,
                                         const TcSmem& sm, int* rstate) {
    constexpr int NT = 1;   // bf16 terms per input value
    const int H = p.H, E = p.E, T = p.T;
    const int n_sl = H / p.rslice;
    const int n_tb = router_tblocks(p);
    const int r = u / n_tb, eg = r / n_sl, sl = r % n_sl;
    const int tbeg = (u % n_tb) * p.rtok, tend = min(T, tbeg + p.rtok);   // this unit's tokens
    const int c0 = sl * p.rslice;
    const int ncols = p.rslice;                          // 256, 512 or 1024
    const int G = router_groups(p), TP = kPRouteTok * G;  // token groups / tokens per pass
    const int wpg = 16 / G;                              // warps per token group (split K)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = warp / wpg, kp = warp % wpg;          // this warp's token group and K part
    const int ne = min(kPRouteExperts, E - eg * kPRouteExperts);
    const uint32_t stride = router_stride(p), wbase = router_wbase(p);
    uint8_t* xt = sm.slots;                              // [8 G][stride]: row 8 g + t = token t of group g
    float* red = reinterpret_cast<float*>(sm.slots);     // [16 warps][32 experts][24] after the MMAs
    int* flag = rstate + 4;
    auto rs = [&](int i) {   // router timestamps of unit 0, or 1 with token blocks (CTA 0's second unit; profiling)
        if (u == (n_tb > 1 ? 1 : 0) && l == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[48 + i] = globaltimer_ns();
    };
    rs(0);
    fence_proxy_async_shared();
    __syncthreads();   // earlier users of the slot area are done
    if (threadIdx.x == 0) {
        const bool pre = rstate[2] == u && rstate[3] == l;
        // the previous unit's weights are this unit's (same slice and layer; they landed in that unit)
        const bool resident = !pre && rstate[5] == r && rstate[6] == l;
        rstate[2] = rstate[3] = -1;
        rstate[8] = !pre && !resident;
        rstate[10] = pre && rstate[9];   // this unit's input rows were copied with its weights
        rstate[9] = 0;
    }
    __syncthreads();
    if (rstate[8]) router_fetch(p, ly, u, sm);
    const bool x_pre = rstate[10] != 0;
    const uint32_t xs_a = smem_u32(xt), ws_a = smem_u32(sm.slots + wbase);
    for (int t0 = tbeg; t0 < tend; t0 += TP) {
        const int nt = min(TP, tend - t0);
        if (t0 > tbeg) __syncthreads();   // the previous pass's sums have been read
        if (t0 == tbeg) rs(1);
        // the pass's rows of x as they are (rows >= nt keep stale data: their output
        // columns are not stored); already in flight when issued with the weights
        const int n16 = ncols / 8;   // 16-byte pieces per row
        for (int i = x_pre ? nt * n16 : threadIdx.x; i < nt * n16; i += blockDim.x) {
            const int t = i / n16, c = (i % n16) * 8;
            cp_async_16(xs_a + (uint32_t)t * stride + (uint32_t)c * 2, p.x + (size_t)(t0 + t) * H + c0 + c);
        }
        cp_async_wait_all();   // this thread's weight and input copies have landed
        __syncthreads();
        if (t0 == tbeg && threadIdx.x == 0) {
            rstate[5] = r;   // weight slice now in shared memory
            rstate[6] = l;
        }
        if (t0 == tbeg) rs(2);
        // this warp's K part: ncols / wpg columns in steps of 16, against its group's 8 NT rows
        float d[2][NT][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < NT; ++b)
#pragma unroll
                for (int q = 0; q < 4; ++q) d[a][b][q] = 0.0f;
        const int kw = ncols / wpg;
        const uint32_t xg = xs_a + (uint32_t)(8 * NT * gw) * stride;
        for (int ks = 0; ks < kw; ks += 16) {
            const int k0 = kp * kw + ks;
            uint32_t af[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
                ldmatrix_x4(ws_a + (uint32_t)(mt * 16 + (lane & 15)) * stride + (uint32_t)(k0 + (lane >> 4) * 8) * 2,
                            af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
            uint32_t b[NT][2];
            ldmatrix_x2(xg + (uint32_t)(8 * (NT - 1) + (lane & 7)) * stride + (uint32_t)(k0 + ((lane >> 3) & 1) * 8) * 2,
                        b[NT - 1][0], b[NT - 1][1]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nb = 0; nb < NT; ++nb)
                    mma_bf16_16816(d[mt][nb], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b[nb][0], b[nb][1]);
        }
        __syncthreads();   // every warp's reads of the x terms are done: red overwrites them
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nb = 0; nb < NT; ++nb) {
                const int e = mt * 16 + (lane >> 2), n = nb * 8 + 2 * (lane & 3);
                float* r = red + warp * 768;
                r[e * 24 + n] = d[mt][nb][0];
                r[e * 24 + n + 1] = d[mt][nb][1];
                r[(e + 8) * 24 + n] = d[mt][nb][2];
                r[(e + 8) * 24 + n + 1] = d[mt][nb][3];
            }
        __syncthreads();
        for (int i = threadIdx.x; i < kPRouteExperts * TP; i += blockDim.x) {   // (expert, token): K parts in order, then the terms
            const int e = i / TP, t = i % TP, g = t >> 3, t8 = t & 7;
            float sh = 0.0f;
            for (int w = 0; w < wpg; ++w) sh += red[(g * wpg + w) * 768 + e * 24 + t8];
            if (t < nt && e < ne) p.rpart[((size_t)sl * T + t0 + t) * E + eg * kPRouteExperts + e] = sh;
        }
        if (t0 == tbeg) rs(3);
    }
    rs(4);
    if (!route_is_small(p)) return;   // larger blocks: the grid sums the partials (logits_reduce)
    // the last unit of the group turns the slice partials into logits
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int old = atomicAdd(p.rcnt + l * 32 + eg, 1);
        *flag = old == n_sl - 1;
        if (old == n_sl - 1) atomicExch(p.rcnt + l * 32 + eg, 0);   // every unit counted: back to rest
        __threadfence();
    }
    __syncthreads();
    if (*flag) {
        for (int i = threadIdx.x; i < T * kPRouteExperts; i += blockDim.x) {
            const int t = i / kPRouteExperts, e = eg * kPRouteExperts + i % kPRouteExperts;
            if (i % kPRouteExperts >= ne) continue;
            const float* src = p.rpart + (size_t)t * E + e;
            float z = 0.0f;
            for (int s0 = 0; s0 < n_sl; s0 += 8) {   // 8 loads in flight, summed in slice order
                float a[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] = s0 + q < n_sl ? __ldcg(src + (size_t)(s0 + q) * T * E) : 0.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (s0 + q < n_sl) z += a[q];
            }
            p.rb.logits[(size_t)t * E + e] = z + (ly.router_b ? __ldg(ly.router_b + e) : 0.0f);
        }
    }
}

// Whole-row router units (a single layer on a block of at most 8 tokens, when x and a
// unit's weight rows fit in shared memory): unit u = experts [u F, u F + F) over all H
// columns, so every logit is complete inside one CTA and no cross-CTA sum is needed.
// Shared memory (slot area): x [T rows][H * 2 + 16 B] at 0, the unit's weight rows at
// router_full_wbase (rows padded by 16 bytes: conflict-free ldmatrix).
__device__ __forceinline__ uint32_t router_full_stride(const PersistParams& p) { return (uint32_t)p.H * 2 + 16; }
__device__ __forceinline__ uint32_t router_full_wbase(const PersistParams& p) {
    return ((uint32_t)p.T * router_full_stride(p) + 1023u) & ~1023u;
}
__device__ __forceinline__ int router_full_units(const PersistParams& p) { return (p.E + p.rfull - 1) / p.rfull; }
// The copies of unit u (x and its weight rows), 16-byte cp.async over the whole CTA.
__device__ __forceinline__ void router_full_fetch(const PersistParams& p, const PersistLayer& ly, int u,
                                                  const TcSmem& sm) {
    const int n16 = p.H / 8, e0 = u * p.rfull, ne = min(p.rfull, p.E - e0);
    const uint32_t stride = router_full_stride(p), xs = smem_u32(sm.slots), wsb = xs + router_full_wbase(p);
    const uint64_t pol = l2_evict_first_policy();
    for (int i = threadIdx.x; i < ne * n16; i += blockDim.x) {
        const int r = i / n16, c = (i % n16) * 8;
        cp_async_16_hint(wsb + (uint32_t)r * stride + (uint32_t)c * 2, ly.router_w + (size_t)(e0 + r) * p.H + c, pol);
    }
    for (int i = threadIdx.x; i < p.T * n16; i += blockDim.x) {
        const int t = i / n16, c = (i % n16) * 8;
        cp_async_16(xs + (uint32_t)t * stride + (uint32_t)c * 2, p.x + (size_t)t * p.H + c);
    }
}
// logit[t][e] = sum_h x[t,h] Wr[e,h] + b[e] for the unit's experts: the 16 warps split
// H, each with mma.sync m16n8k16 (rows = experts, columns = tokens; bf16 products are
// exact, fp32 sums), then the warps' partial sums are added in warp order.
__device__ __noinline__ void router_full_unit(const PersistParams& p, const PersistLayer& ly, int u, const TcSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = u * p.rfull, ne = min(p.rfull, p.E - e0);
    const uint32_t stride = router_full_stride(p), xs = smem_u32(sm.slots), wsb = xs + router_full_wbase(p);
    const bool writer = threadIdx.x < ne * p.T;   // thread (e, t) writes logit[t][e0 + e]
    const float bias = writer && ly.router_b ? __ldg(ly.router_b + e0 + threadIdx.x / p.T) : 0.0f;   // loaded early
    cp_async_wait_all();
    __syncthreads();
    const int kw = p.H / 16;                                   // columns per warp (multiple of 16)
    const int arow = min(lane & 15, ne - 1), brow = min(lane & 7, p.T - 1);   // rows past the unit / block: repeats
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < kw; ks += 16) {
        const int k0 = warp * kw + ks;
        uint32_t a0, a1, a2, a3, b0, b1;
        ldmatrix_x4(wsb + (uint32_t)arow * stride + (uint32_t)(k0 + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
        ldmatrix_x2(xs + (uint32_t)brow * stride + (uint32_t)(k0 + ((lane >> 3) & 1) * 8) * 2, b0, b1);
        mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
    }
    // the warps' sums go to the scale ring (unused until the expert phase), so that x stays
    // in the slot area for operand_tasks
    float* red = reinterpret_cast<float*>(sm.scales);          // [16 warps][16 experts][8 tokens]
    {
        const int e = lane >> 2, t = 2 * (lane & 3);
        red[(warp * 16 + e) * 8 + t] = d[0];
        red[(warp * 16 + e) * 8 + t + 1] = d[1];
        red[(warp * 16 + e + 8) * 8 + t] = d[2];
        red[(warp * 16 + e + 8) * 8 + t + 1] = d[3];
    }
    __syncthreads();
    if (writer) {
        const int e = threadIdx.x / p.T, t = threadIdx.x % p.T;
        float z = 0.0f;
        for (int w = 0; w < 16; ++w) z += red[(w * 16 + e) * 8 + t];
        p.rb.logits[(size_t)t * p.E + e0 + e] = z + bias;
    }
}

// Logits of a larger block from the router slice partials (slices in order) + bias,
// over every thread of the grid.  Residual stack: the partials are the router products
// of r * w_norm per 256-column block (prep_unit), times 1 / rms(r_t), which is also
// written to tscale[t] for the gate/up epilogue.
__device__ __noinline__ void logits_reduce(const PersistParams& p, const PersistLayer& ly) {
    const int TE = p.T * p.E, n_sl = p.norm ? p.H / kCombineChunk : p.H / p.rslice;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < TE; i += gridDim.x * blockDim.x) {
        float iv = 1.0f;
        if (p.norm) {   // the sum of the token's block sums of squares in block order, as inv_rms
            const int t = i / p.E, nc = p.H / kCombineChunk;
            float tot = 0.0f;
            for (int c = 0; c < nc; ++c) tot += __ldcg(p.ss + (size_t)t * nc + c);
            iv = 1.0f / sqrtf(tot / (float)p.H + p.eps);
            if (i % p.E == 0) p.tscale[t] = iv;
        }
        const float* src = p.rpart + i;
        float z = 0.0f;
        for (int s0 = 0; s0 < n_sl; s0 += 8) {   // 8 loads in flight, summed in slice order
            float a[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) a[q] = s0 + q < n_sl ? __ldcg(src + (size_t)(s0 + q) * TE) : 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (s0 + q < n_sl) z += a[q];
        }
        p.rb.logits[i] = (p.norm ? z * iv : z) + (ly.router_b ? __ldg(ly.router_b + i % p.E) : 0.0f);
    }
}

// The expert operand of the layer input x (a residual stack forms its operand in
// prep_unit): task i = (token t, MX block kb) splits the block's 32 values into 8 E2M1
// terms.  Whole warps;
// the tasks are spread over every warp of the grid, starting from the last CTA
// (the first CTAs run the router units).
// xsm: this CTA's shared-memory copy of x (rows of router_full_stride bytes; a whole-row
// router unit's input), or NULL.
__device__ __noinline__ void operand_tasks(const PersistParams& p, const PersistLayer& ly, const uint8_t* xsm) {
    const int H = p.H, nb = H / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int gw = (gridDim.x - 1 - blockIdx.x) * nw + warp;
    const int n = p.T * nb, step = gridDim.x * nw;
    if (n <= step) {   // at most one task per warp (small blocks): the short code path
        if (gw < n) {
            const int t = gw / nb, kb = gw % nb;
            const size_t o = (size_t)t * H + kb * 32 + lane;
            const float v = xsm ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(
                                      xsm + (size_t)t * router_full_stride(p))[kb * 32 + lane])
                                : __bfloat162float(p.x[o]);
            uint32_t sb0, sb1;
            const uint32_t codes = split_e2m1_terms(v, sb0, sb1);
            store_act_terms(p.xb4, p.xsf, H, t, kb, lane, codes, sb0, sb1);
        }
        fence_proxy_async_global();
        return;
    }
    constexpr int kB = 4;   // tasks in flight per warp: their loads and shuffle chains overlap
    for (int i0 = gw; i0 < n; i0 += kB * step) {
        float v[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int i = i0 + j * step, t = i / nb, kb = i % nb;
            v[j] = 0.0f;
            if (i >= n) continue;
            const size_t o = (size_t)t * H + kb * 32 + lane;
            v[j] = __bfloat162float(p.x[o]);
        }
        uint32_t codes[kB], sb0[kB], sb1[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) codes[j] = split_e2m1_terms<true>(v[j], sb0[j], sb1[j]);
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int i = i0 + j * step;
            if (i < n) store_act_terms(p.xb4, p.xsf, H, i / nb, i % nb, lane, codes[j], sb0[j], sb1[j]);
        }
    }
    fence_proxy_async_global();   // read next by the expert phase's bulk copies
}

// Orderable key of a logit for unsigned max: larger logits give larger keys; NaN
// ranks with -inf.  Key 0 is below every logit (used for taken / absent entries).
__device__ __forceinline__ uint32_t logit_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (v != v) u = 0xFF800000u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k + gates of one token's logits row, by one warp: lane l owns experts l, l + 32,
// ...; each round takes the largest key (redux max), the lowest expert among equal keys
// (redux min), and the winning lane moves to its next candidate.  For k <= 8 every lane
// keeps its own 8 best (key desc, expert asc) sorted in registers; for larger k the
// winning lane rescans its experts.  Lane j < k returns pick j and its gate (softmax
// over the k selected logits).  kGlobal: the row is in global memory (read from L2).
template <bool kGlobal>
__device__ __forceinline__ void topk_warp(const float* row, int E, int k, int lane, uint32_t& mine, float& gate) {
    auto ld = [&](int e) -> float { return kGlobal ? __ldcg(row + e) : row[e]; };
    mine = 0u;
    if (k <= 8) {
        uint32_t kk[8], ee[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) { kk[i] = 0u; ee[i] = 0xFFFFFFFFu; }
#pragma unroll 4
        for (int e = lane; e < E; e += 32) {
            uint32_t ck = logit_key(ld(e)), ce = (uint32_t)e;
#pragma unroll
            for (int i = 0; i < 8; ++i) {   // keep the larger here, carry the smaller down
                const bool gt = ck > kk[i];
                const uint32_t tk = gt ? kk[i] : ck, te = gt ? ee[i] : ce;
                kk[i] = gt ? ck : kk[i];
                ee[i] = gt ? ce : ee[i];
                ck = tk;
                ce = te;
            }
        }
        for (int j = 0; j < k; ++j) {
            const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, kk[0]);
            const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, kk[0] == kmax ? ee[0] : 0xFFFFFFFFu);
            if (lane == j) mine = emin;
            if (ee[0] == emin) {
#pragma unroll
                for (int i = 0; i < 7; ++i) { kk[i] = kk[i + 1]; ee[i] = ee[i + 1]; }
                kk[7] = 0u;
                ee[7] = 0xFFFFFFFFu;
            }
        }
    } else {
        uint32_t taken = 0u;
        uint32_t bk = 0u;
        uint32_t be = 0xFFFFFFFFu;
        auto rescan = [&]() {
            bk = 0u;
            be = 0xFFFFFFFFu;
            for (int i = 0, e = lane; e < E; ++i, e += 32) {
                const uint32_t kk = ((taken >> i) & 1u) ? 0u : logit_key(ld(e));
                if (kk > bk) { bk = kk; be = (uint32_t)e; }
            }
        };
        rescan();
        for (int j = 0; j < k; ++j) {
            const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bk);
            const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, bk == kmax ? be : 0xFFFFFFFFu);
            if (lane == j) mine = emin;
            if ((int)(emin & 31u) == lane) {
                taken |= 1u << (emin >> 5);
                rescan();
            }
        }
    }
    float v = lane < k ? ld((int)mine) : 0.0f;
    if (v != v) v = __int_as_float(0xFF800000);
    const float m = __shfl_sync(0xFFFFFFFFu, v, 0);
    const float ex = lane < k ? expf(v - m) : 0.0f;
    const float den = warp_sum(ex);
    gate = ex / den;
}

// Top-k + gates of every token of a larger block, one warp per token over the whole
// grid, into the workspace (idx / gate).
__device__ __noinline__ void topk_tokens(const PersistParams& p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int t = blockIdx.x * nw + warp; t < p.T; t += gridDim.x * nw) {
        uint32_t mine;
        float gate;
        topk_warp<true>(p.rb.logits + (size_t)t * p.E, p.E, p.k, lane, mine, gate);
        if (lane < p.k) {
            p.rb.idx[t * p.k + lane] = (int)mine;
            p.rb.gate[t * p.k + lane] = gate;
        }
    }
}

// Routing of a small verify block (T*k <= 64, T*E <= 8192) by every CTA into its own
// shared memory: the layer's logits, top-k + gates, and the grouping as a routing
// table for the expert phase and the combine.  Every CTA computes the same values.
// scratch: >= T*E + 2*E + 64 ints of shared memory.
__device__ __noinline__ void route_small(const PersistParams& p, int l, int* scratch, RouteTable* rt) {
    const int T = p.T, E = p.E, k = p.k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    auto sub = [&](int i) {   // sub-step timestamps of the first layer, CTA 0 (profiling)
        if (l == 0 && blockIdx.x == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[40 + i] = globaltimer_ns();
    };
    sub(0);
    float* lg = reinterpret_cast<float*>(scratch);   // [T * E]
    int* cnt = scratch + T * E;                      // [E]
    int* off = cnt + E;                              // [E]
    int* wsum = off + E;                             // [32 + 4]
    int* cnt0 = wsum + 36;                           // [E] pairs among the first 32 per expert
    const int n = T * E;
    if (p.norm) {
        // residual stack: logit[t][e] = (1 / rms(r_t)) * sum over column blocks of the
        // router products of r * w_norm (prep_unit), in block order, + bias
        for (int t = warp; t < T; t += nw) {
            const float iv = inv_rms(p, t);
            if (lane == 0) rt->tscale[t] = iv;
        }
        __syncthreads();
        const PersistLayer& ly = p.layer[l];
        const int nc = p.H / kCombineChunk;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float* src = p.rpart + i;
            float z = 0.0f;
            for (int c0 = 0; c0 < nc; c0 += 8) {   // 8 loads in flight, summed in block order
                float a[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] = c0 + q < nc ? __ldcg(src + (size_t)(c0 + q) * n) : 0.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (c0 + q < nc) z += a[q];
            }
            lg[i] = z * rt->tscale[i / E] + (ly.router_b ? __ldg(ly.router_b + i % E) : 0.0f);
        }
    } else {
        for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {   // 8 loads in flight per thread
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + q * blockDim.x;
                v[q] = i < n ? __ldcg(p.rb.logits + i) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + q * blockDim.x;
                if (i < n) lg[i] = v[q];
            }
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        cnt[e] = 0;
        cnt0[e] = 0;
    }
    __syncthreads();
    sub(1);
    for (int t = warp; t < T; t += nw) {
        uint32_t mine;
        float gate;
        topk_warp<false>(lg + (size_t)t * E, E, k, lane, mine, gate);
        if (lane < k) {
            rt->idx[t * k + lane] = (int)mine;
            rt->gate[t * k + lane] = gate;
        }
    }
    __syncthreads();
    sub(2);
    const int npairs = T * k;
    for (int s = threadIdx.x; s < npairs; s += blockDim.x) {
        const int e = rt->idx[s];
        if (e >= p.e_begin && e < p.e_end) {
            atomicAdd(&cnt[e], 1);
            if (s < 32) atomicAdd(&cnt0[e], 1);
        }
    }
    __syncthreads();
    // exclusive scans over the experts of (pairs, routed flag), packed in 16-bit
    // halves (both totals <= 64); thread i owns experts 2i and 2i + 1
    {
        const int ea = 2 * threadIdx.x, eb = ea + 1;
        const int ca = ea < E ? cnt[ea] : 0, cb = eb < E ? cnt[eb] : 0;
        const int va = (ca << 16) | (ca > 0 ? 1 : 0), vb = (cb << 16) | (cb > 0 ? 1 : 0);
        int incl = va + vb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int s = lane < nw ? wsum[lane] : 0;
            int si = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, si, o);
                if (lane >= o) si += u;
            }
            if (lane < nw) wsum[lane] = si - s;
            if (lane == 31) wsum[32] = si;
        }
        __syncthreads();
        const int xa = wsum[warp] + incl - va - vb, xb = xa + va;
        if (ea < E) {
            off[ea] = xa >> 16;
            if (ca > 0) {
                rt->e[xa & 0xFFFF] = ea;
                rt->beg[xa & 0xFFFF] = xa >> 16;
                rt->cnt[xa & 0xFFFF] = ca;
            }
        }
        if (eb < E) {
            off[eb] = xb >> 16;
            if (cb > 0) {
                rt->e[xb & 0xFFFF] = eb;
                rt->beg[xb & 0xFFFF] = xb >> 16;
                rt->cnt[xb & 0xFFFF] = cb;
            }
        }
    }
    __syncthreads();
    sub(3);
    const int n_active = wsum[32] & 0xFFFF, n_in = wsum[32] >> 16;
    if (warp == 0) {   // first chunk of each routed expert (<= 64 of them; lane owns 2)
        const int a0 = 2 * lane, a1 = a0 + 1;
        const int h0 = a0 < n_active ? (rt->cnt[a0] + kTmaTok - 1) / kTmaTok : 0;
        const int h1 = a1 < n_active ? (rt->cnt[a1] + kTmaTok - 1) / kTmaTok : 0;
        int incl = h0 + h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += u;
        }
        if (a0 < n_active) rt->chunk0[a0] = incl - h0 - h1;
        if (a1 < n_active) rt->chunk0[a1] = incl - h1;
        if (lane == 31) {
            rt->n_active = n_active;
            rt->n_chunks = incl;
            rt->pad0 = n_in;   // pairs routed into the shard
        }
    }
    // perm position of pair s (< 64: warps 0 and 1): its expert's offset + the same-expert
    // pairs before it, i.e. the lower lanes of its warp with the same expert (match) and,
    // in warp 1, the first 32 pairs' count of that expert
    if (threadIdx.x < 64) {
        const int s = threadIdx.x;
        const int e = s < npairs ? rt->idx[s] : -1 - s;   // (absent pairs match nothing)
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        if (s < npairs && e >= p.e_begin && e < p.e_end) {
            const int r = __popc(same & ((1u << lane) - 1u)) + (s >= 32 ? cnt0[e] : 0);
            rt->tok[off[e] + r] = s / k;
            rt->pair[off[e] + r] = s;
        }
    }
    __syncthreads();
    sub(4);
}

// The routing of a small verify block, published by one CTA from its routing table:
// idx / gates / counts / offsets / perm / active list (the logits are already in the
// workspace), and the optional per-layer copies.  Called after that CTA's expert phase.
__device__ __noinline__ void publish_small(const PersistParams& p, int l, const RouteTable* rt) {
    const int T = p.T, E = p.E, k = p.k, npairs = T * k;
    const RouteBufs& rb = p.rb;
    const int na = rt->n_active, n_in = rt->pad0;
    const int lgi = p.layer_base + l;
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
        const int perm = i < n_in ? rt->pair[i] : -1;
        rb.idx[i] = rt->idx[i];
        rb.gate[i] = rt->gate[i];
        rb.perm[i] = perm;
        if (p.dbg.idx) p.dbg.idx[(size_t)lgi * npairs + i] = rt->idx[i];
        if (p.dbg.gate) p.dbg.gate[(size_t)lgi * npairs + i] = rt->gate[i];
        if (p.dbg.perm) p.dbg.perm[(size_t)lgi * npairs + i] = perm;
    }
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        int lo = 0, hi = na;   // first routed expert with id >= e
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (rt->e[mid] < e) lo = mid + 1; else hi = mid;
        }
        const int offs = lo < na ? rt->beg[lo] : n_in;
        const int c = (e < E && lo < na && rt->e[lo] == e) ? rt->cnt[lo] : 0;
        rb.offsets[e] = offs;
        if (p.dbg.offsets) p.dbg.offsets[(size_t)lgi * (E + 1) + e] = offs;
        if (e < E) {
            rb.counts[e] = c;
            if (p.dbg.counts) p.dbg.counts[(size_t)lgi * E + e] = c;
        }
    }
    for (int a = threadIdx.x; a < na; a += blockDim.x) rb.active[1 + a] = rt->e[a];
    if (threadIdx.x == 0) rb.active[0] = na;
}

// The next layer's inputs from 256 columns of a token's residual (residual stack).
// RMSNorm(r) = (r * w_norm) / rms(r), and 1 / rms(r) is one factor per token: it is
// applied to the router's logits (route_small / logits_reduce) and to the gate/up
// outputs (tc_epilogue), so what is formed here, column block by column block, is
// y = r * w_norm: its E2M1 terms (the experts' input operand, as operand_tasks stores
// them) and its router products P[cb][t][e] = sum over the block's columns of
// y[h] * W_router[e][h] (fp32, in a fixed order), kept in rpart.  Thread i < 64 holds
// r[4i .. 4i + 3] of block cb in v (have); ys: 256 floats of shared memory.
__device__ __noinline__ void prep_unit(const PersistParams& p, const PersistLayer& lyn, int t, int cb, float4 v,
                                       bool have, float* ys) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = cb * kCombineChunk;
    __syncthreads();   // an earlier unit's reads of ys are done
    if (have) {
        const int h = threadIdx.x * 4;
        const uint2 wv = __ldg(reinterpret_cast<const uint2*>(lyn.norm_w + c0 + h));
        *reinterpret_cast<float4*>(ys + h) =
            make_float4(v.x * bf16_lo(wv.x), v.y * bf16_hi(wv.x), v.z * bf16_lo(wv.y), v.w * bf16_hi(wv.y));
    }
    __syncthreads();
    if (warp < kCombineChunk / 32) {   // the expert operand: MX block c0 / 32 + warp (lane = element)
        uint32_t sb0, sb1;
        const uint32_t codes = split_e2m1_terms(ys[warp * 32 + lane], sb0, sb1);
        store_act_terms(p.xb4, p.xsf, p.H, t, c0 / 32 + warp, lane, codes, sb0, sb1);
    }
    // router products: warp w takes experts w, w + 16, ...; lane l the columns 8l .. 8l + 7
    const float4 y0 = *reinterpret_cast<const float4*>(ys + lane * 8);
    const float4 y1 = *reinterpret_cast<const float4*>(ys + lane * 8 + 4);
    for (int e = warp; e < p.E; e += blockDim.x >> 5) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(lyn.router_w + (size_t)e * p.H + c0 + lane * 8));
        float z = y0.x * bf16_lo(w.x);
        z = fmaf(y0.y, bf16_hi(w.x), z);
        z = fmaf(y0.z, bf16_lo(w.y), z);
        z = fmaf(y0.w, bf16_hi(w.y), z);
        z = fmaf(y1.x, bf16_lo(w.z), z);
        z = fmaf(y1.y, bf16_hi(w.z), z);
        z = fmaf(y1.z, bf16_lo(w.w), z);
        z = fmaf(y1.w, bf16_hi(w.w), z);
        z = warp_sum(z);
        if (lane == 0) p.rpart[((size_t)cb * p.T + t) * p.E + e] = z;
    }
    fence_proxy_async_global();   // the operand is read next by bulk copies
}

// Combine unit (token t, 256-column block c): out = sum_j gate[t, j] * partial[t*k + j]
// (slots in order, pairs outside the expert shard skipped); with a residual stack
// r += out and the block's sum of squares of r is kept for the next RMSNorm, and when
// the next layer runs in this launch its inputs are prepared from r (prep_unit).  The
// last layer writes y.
// dry: read everything but store nothing (runs the code once to bring it into the caches).
__device__ __noinline__ void combine_unit(const PersistParams& p, int u, int l, float* red, const RouteTable* rt,
                                          float* ys, bool dry = false) {
    const int H = p.H, k = p.k;
    const int nc = H / kCombineChunk;
    const int t = u / nc, c = u % nc;
    const int c0 = c * kCombineChunk, ncols = kCombineChunk;
    const RouteBufs& rb = p.rb;
    const bool last = l == p.L - 1;
    const size_t o = (size_t)t * H + c0;
    float gj[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {   // gates of the slots in the shard (0 outside)
        gj[j] = 0.0f;
        if (j < k) {
            const int e = rt ? rt->idx[t * k + j] : __ldcg(rb.idx + t * k + j);
            const float g = rt ? rt->gate[t * k + j] : __ldcg(rb.gate + t * k + j);
            gj[j] = (e >= p.e_begin && e < p.e_end) ? g : 0.0f;
        }
    }
    float ssl = 0.0f;
    const int h = threadIdx.x * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < ncols) {
#pragma unroll
        for (int j0 = 0; j0 < kMaxTopK; j0 += 8) {   // 8 slots' loads in flight, summed in slot order
            if (j0 >= k) break;
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = j0 + q;
                v[q] = (j < k && gj[j] != 0.0f)
                           ? __ldcg(reinterpret_cast<const float4*>(p.ta.partial + (size_t)(t * k + j) * H + c0 + h))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = j0 + q;
                if (j < k && gj[j] != 0.0f) {
                    acc.x = fmaf(gj[j], v[q].x, acc.x);
                    acc.y = fmaf(gj[j], v[q].y, acc.y);
                    acc.z = fmaf(gj[j], v[q].z, acc.z);
                    acc.w = fmaf(gj[j], v[q].w, acc.w);
                }
            }
        }
        if (p.norm) {
            const float4 r = __ldcg(reinterpret_cast<const float4*>(p.resid + o + h));
            acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
            if (!dry) *reinterpret_cast<float4*>(p.resid + o + h) = acc;
            ssl = acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
        }
        if (last && p.write_y && !dry) {
            if (p.y_bf16) {
                __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 v;
                v.x = *reinterpret_cast<uint32_t*>(&a);
                v.y = *reinterpret_cast<uint32_t*>(&b);
                *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o + h) = v;
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o + h) = acc;
            }
        }
    }
    if (p.norm) {
        const float tot = block_sum(ssl, red);
        if (threadIdx.x == 0 && !dry) p.ss[(size_t)t * nc + c] = tot;
        if (!dry && l + 1 < p.L) prep_unit(p, p.layer[l + 1], t, c, acc, h < ncols, ys);
    }
}

// Start of a launch of a residual stack, unit (token t, 256-column block c): the residual
// (r = fp32(x) on the first launch of the stack, stored; else the residual left by the
// previous launch), its block sum of squares, and the first layer's inputs (prep_unit).
__device__ __noinline__ void stack_prep_unit(const PersistParams& p, int u, float* red, float* ys) {
    const int H = p.H;
    const int nc = H / kCombineChunk;
    const int t = u / nc, c = u % nc;
    const size_t o = (size_t)t * H + (size_t)c * kCombineChunk;
    float ssl = 0.0f;
    const int h = threadIdx.x * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < kCombineChunk) {
        if (p.init_from_x) {
            const uint2 xv = __ldg(reinterpret_cast<const uint2*>(p.x + o + h));
            v = make_float4(bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y));
            *reinterpret_cast<float4*>(p.resid + o + h) = v;
        } else {
            v = __ldcg(reinterpret_cast<const float4*>(p.resid + o + h));
        }
        ssl = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    const float tot = block_sum(ssl, red);
    if (threadIdx.x == 0) p.ss[(size_t)t * nc + c] = tot;
    prep_unit(p, p.layer[0], t, c, v, h < kCombineChunk, ys);
}


// Grouping of a larger block by one CTA (after topk_tokens): counts, offsets, perm,
// the routed-expert list and each routed expert's first chunk, published in the
// workspace for the work-list builders (build_items_slice).
// scratch: shared memory of at least (2 * E + 1 + 32 * E + 64 + T * k + 2 * E) ints (the
// pairs' experts, the counts and the active list are read from it, not from the workspace).
static_assert((36 * kMaxExperts + 65 + 512 * kTmaTok) * sizeof(int) <=
                  (size_t)TcWide::kStages * TcWide::kSlotBytes + kTcScaleRing * TcWide::kScaleEntry,
              "the grouping's shared-memory arrays fit the slot area and the scale ring");
__device__ __noinline__ void route_phase(const PersistParams& p, const PersistLayer& ly, int l, int* scratch) {
    const int T = p.T, E = p.E, k = p.k, H = p.H;
    const RouteBufs& rb = p.rb;
    const WorkList& wl = p.wl;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    auto sub = [&](int i) {   // sub-step timestamps of the first layer (profiling)
        if (l == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[40 + i] = globaltimer_ns();
    };
    sub(0);
    // (top-k and gates were written by topk_tokens)
    sub(1);
    const int npairs = T * k;
    int* cnt = scratch;                  // [E] counts, then offsets
    int* flag = scratch + E;             // [E + 1]
    int* wcnt = scratch + 2 * E + 1;     // [32][E] (nw <= 32)
    int* misc = wcnt + 32 * E;           // [64]
    int* sidx = misc + 64;               // [T * k] each pair's expert, -1 outside the shard
    int* scnt = sidx + npairs;           // [E] counts
    int* sact = scnt + E;                // [E] the active list
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < npairs; s += blockDim.x) {
        int e = rb.idx[s];
        if (e < p.e_begin || e >= p.e_end) e = -1;
        sidx[s] = e;
        if (e >= 0) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    sub(2);
    // ---- counts, offsets, active list (warp 0)
    if (warp == 0) {
        for (int e = lane; e < E; e += 32) {
            rb.counts[e] = cnt[e];
            scnt[e] = cnt[e];
            flag[e] = cnt[e] > 0 ? 1 : 0;
        }
        __syncwarp();
        const int total = warp_excl_scan(cnt, E);            // cnt -> offsets
        __syncwarp();
        const int n_active = warp_excl_scan(flag, E);        // flag -> active position
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            rb.offsets[e] = cnt[e];
            if (scnt[e] > 0) {
                rb.active[1 + flag[e]] = e;
                sact[flag[e]] = e;
            }
        }
        if (lane == 0) {
            rb.offsets[E] = total;
            rb.active[0] = n_active;
            misc[0] = n_active;
        }
    }
    __syncthreads();
    // ---- perm: pairs in id order inside each expert.  Warp w owns the contiguous segment
    // [w seg, (w + 1) seg) of the pair ids: its per-expert counts, one scan over the warps
    // in warp order (on top of the expert offsets), then each warp places its pairs in order.
    const int seg = (npairs + nw - 1) / nw;
    const int s_lo = min(npairs, warp * seg), s_hi = min(npairs, s_lo + seg);
    auto pair_expert = [&](int s) { return s < s_hi ? sidx[s] : -1; };
    for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    for (int b = s_lo; b < s_hi; b += 32) {
        const int e = pair_expert(b + lane);
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && (peers & ((1u << lane) - 1u)) == 0) wcnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int run = cnt[x];
        for (int w = 0; w < nw; ++w) {
            const int c = wcnt[w * E + x];
            wcnt[w * E + x] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int b = s_lo; b < s_hi; b += 32) {
        const int s = b + lane, e = pair_expert(s);
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const int lane_rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0) rb.perm[wcnt[warp * E + e] + lane_rank] = s;
        __syncwarp();
        if (e >= 0 && lane_rank == 0) wcnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    sub(3);
    // ---- first chunk of each routed expert (chunks of <= p.chunk pairs) and the item counts
    const int n_active = misc[0];
    const int rbu = p.I / kTmaRows, rbd = H / kDownRows;
    int* chunk0 = flag;                 // [n_active + 1]
    for (int a = threadIdx.x; a < n_active; a += blockDim.x) chunk0[a] = (scnt[sact[a]] + p.chunk - 1) / p.chunk;
    __syncthreads();
    if (warp == 0) {
        const int total_chunks = warp_excl_scan(chunk0, n_active);
        if (lane == 0) {
            chunk0[n_active] = total_chunks;
            wl.n_items[0] = total_chunks * (rbu + rbd);
            wl.n_items[1] = total_chunks * rbu;
        }
    }
    __syncthreads();
    for (int a = threadIdx.x; a <= n_active; a += blockDim.x) wl.chunk0[a] = chunk0[a];
    sub(4);
    // ---- optional copies of the routing
    const int lg = p.layer_base + l;
    if (p.dbg.idx) for (int i = threadIdx.x; i < T * k; i += blockDim.x) p.dbg.idx[(size_t)lg * T * k + i] = rb.idx[i];
    if (p.dbg.gate) for (int i = threadIdx.x; i < T * k; i += blockDim.x) p.dbg.gate[(size_t)lg * T * k + i] = rb.gate[i];
    if (p.dbg.perm) for (int i = threadIdx.x; i < T * k; i += blockDim.x) p.dbg.perm[(size_t)lg * T * k + i] = rb.perm[i];
    if (p.dbg.counts) for (int i = threadIdx.x; i < E; i += blockDim.x) p.dbg.counts[(size_t)lg * E + i] = rb.counts[i];
    if (p.dbg.offsets)
        for (int i = threadIdx.x; i <= E; i += blockDim.x) p.dbg.offsets[(size_t)lg * (E + 1) + i] = rb.offsets[i];
}

// This CTA's share of the work list of a larger block (all CTAs, after the grouping is
// published): items in the order of table_item (per routed expert, row block major,
// chunk minor; gate/up items first).  scratch: 4 * (n_active + 1) ints of shared memory.
__device__ __noinline__ void build_items_slice(const PersistParams& p, int* scratch) {
    const RouteBufs& rb = p.rb;
    const WorkList& wl = p.wl;
    const int k = p.k;
    const int n_active = __ldcg(rb.active);
    int* s_c0 = scratch;                  // [n_active + 1]
    int* s_act = s_c0 + n_active + 1;     // [n_active]
    int* s_beg = s_act + n_active;
    int* s_cnt = s_beg + n_active;
    for (int a = threadIdx.x; a <= n_active; a += blockDim.x) {
        s_c0[a] = __ldcg(wl.chunk0 + a);
        if (a < n_active) {
            const int e = __ldcg(rb.active + 1 + a);
            s_act[a] = e;
            s_beg[a] = __ldcg(rb.offsets + e);
            s_cnt[a] = __ldcg(rb.counts + e);
        }
    }
    __syncthreads();
    const int rbu = p.I / kTmaRows, rbd = p.H / kDownRows;
    const int total_chunks = s_c0[n_active];
    const int n_gu = total_chunks * rbu, total = total_chunks * (rbu + rbd);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const bool down = i >= n_gu;
        const int j = down ? i - n_gu : i;
        const int nrb = down ? rbd : rbu;
        int lo = 0, hi = n_active - 1;   // the routed expert whose items contain j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_c0[mid] * nrb <= j) lo = mid; else hi = mid - 1;
        }
        const int nch = (s_cnt[lo] + p.chunk - 1) / p.chunk;
        const int rr = j - s_c0[lo] * nrb, rbi = rr / nch, tc = rr % nch;   // row block major, chunk minor
        ItemRec r;
        r.code = item_code(down ? kItemDown : kItemGateUp, rbi, tc, lo);
        r.e = s_act[lo];
        r.beg = s_beg[lo] + tc * p.chunk;
        r.ntok = min(p.chunk, s_cnt[lo] - tc * p.chunk);
        // the pairs' ids as 16-bit halves (T * k <= 4096 on this path): word q holds pair
        // slots 2q (low half) and 2q + 1
#pragma unroll
        for (int q = 0; q < kMaxChunk; ++q) {
            const int p0 = 2 * q < r.ntok ? __ldcg(rb.perm + r.beg + 2 * q) : 0;
            const int p1 = 2 * q + 1 < r.ntok ? __ldcg(rb.perm + r.beg + 2 * q + 1) : 0;
            r.tok[q] = down ? (p0 | (p1 << 16)) : ((p0 / k) | ((p1 / k) << 16));
        }
        r.chunk = s_c0[lo] + tc;
        r.pad[0] = nch;
        r.pad[1] = r.pad[2] = 0;
        wl.items[i] = r;
    }
}

// per-warp staging buffers of the gather: in the slot area and the scale ring, which are
// one contiguous span and idle between expert phases
constexpr uint32_t kGatherBufBase = 17408, kGatherBufBytes = 9216;
static_assert(kGatherBufBase + 16 * kGatherBufBytes <=
                  (uint32_t)(TcWide::kStages * TcWide::kSlotBytes + kTcScaleRing * TcWide::kScaleEntry),
              "gather buffers in the slot area and the scale ring");
static_assert(4 * (kMaxExperts + 1) * sizeof(int) <= kGatherBufBase, "routing arrays below the gather buffers");
// The layer input's expert operand gathered per chunk (larger blocks, every CTA, after
// the grouping is published) into the 128-row layout of the wide expert phase: unit =
// (chunk, 256-wide stage, half h), one warp per unit; pair slot p of the chunk gets the
// first p.terms of its token's 8 term rows (rows p.terms * p + j; the first 4 terms of
// the 8-term split are the 4-term split) and their scales; half h holds the pair slots
// h * chunk / 2 .. (rows 64 h .. 64 h + 63).
// scratch: the routing arrays staged by build_items_slice.
__device__ __noinline__ void gather_chunk_operand(const PersistParams& p, const int* scratch, uint8_t* slots) {
    constexpr int kTile = tc_a_tile<TcWide>(), kSfa = tc_sfa_stage<TcWide>();
    const int n_active = __ldcg(p.rb.active);
    const int* s_c0 = scratch;
    const int* s_beg = scratch + n_active + 1 + n_active;
    const int* s_cnt = s_beg + n_active;
    const int nst = p.H / kTcKS, total_chunks = s_c0[n_active];
    const int half = p.chunk / 2;   // pair slots per half (64 rows)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    // this warp's staging buffer: 8 KB of rows + 512 B of scales, past the routing arrays
    const uint32_t buf = smem_u32(slots) + kGatherBufBase + (uint32_t)warp * kGatherBufBytes;
    for (int u = blockIdx.x * nw + warp; u < total_chunks * nst * 2; u += gridDim.x * nw) {
        const int c = u / (2 * nst), st = (u >> 1) % nst, hh = u & 1;
        int lo = 0, hi = n_active - 1;   // the routed expert of chunk c
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_c0[mid] <= c) lo = mid; else hi = mid - 1;
        }
        const int tc = c - s_c0[lo], beg = s_beg[lo] + tc * p.chunk + hh * half;
        const int ntok = min(half, s_cnt[lo] - tc * p.chunk - hh * half);   // <= 0: an empty half
        uint8_t* dst = const_cast<uint8_t*>(p.ta.xc4) + ((size_t)c * nst + st) * kTile + hh * (kTile / 2);   // workspace
        uint8_t* dsf = const_cast<uint8_t*>(p.ta.xcs) + ((size_t)c * nst + st) * kSfa + hh * (kSfa / 2);
        const int rows = p.terms, pp = rows * 8;   // term rows per pair; 16-byte pieces per pair
        // the chunk's tokens (lane q: pair q), then every pair's rows and scales into this
        // warp's shared-memory buffer (all copies in flight at once), then out in one run
        const int tq = lane < ntok ? __ldcg(p.rb.perm + beg + lane) / p.k : 0;
        for (int q = 0; q < ntok; ++q) {
            const int t = __shfl_sync(0xFFFFFFFFu, tq, q);
            const uint8_t* src = p.xb4 + ((size_t)t * nst + st) * 1024;
            for (int i = lane; i < pp; i += 32) cp_async_16(buf + (q * pp + i) * 16, src + i * 16);
            if (lane < rows / 2)
                cp_async_16(buf + 8192 + q * rows * 8 + lane * 16, p.xsf + ((size_t)t * nst + st) * 64 + lane * 16);
        }
        cp_async_wait_all();
        __syncwarp();
        // rows are 128-byte swizzled by their row index mod 8 (the source by term j): with 4
        // terms an odd pair slot's rows 4q + j have phase j ^ 4, so their 16-byte pieces
        // swap places c <-> c ^ 4 (half is even: a slot's parity within the half is its own)
        for (int i = lane; i < ntok * pp; i += 32) {
            const int qq = i / pp, w = i % pp;
            const int o = (rows == 4 && (qq & 1)) ? (w ^ 4) : w;
            reinterpret_cast<int4*>(dst)[qq * pp + o] = ld_shared_v4(buf + i * 16);
        }
        for (int i = lane; i < ntok * rows / 2; i += 32)
            reinterpret_cast<int4*>(dsf)[i] = ld_shared_v4(buf + 8192 + i * 16);
        __syncwarp();   // the buffer is read before the next unit's copies land
    }
}

// y = sum_j g[t, j] * partial[t*k + j] (slot order; slots outside the shard skipped) for
// a layer without a residual stack, over every thread of the grid, 4 columns per step.
// dry: one step per thread of this CTA and nothing stored (brings the code into the caches).
// Blocks routed through the workspace first copy every pair's (expert, gate) into shared
// memory (scratch, up to 4096 pairs), so a step waits for its partials only.
__device__ __noinline__ void combine_elems(const PersistParams& p, int l, const RouteTable* rt, uint8_t* scratch,
                                           bool dry = false) {
    const int H4 = p.H / 4, k = p.k;
    const int n = p.T * H4;
    const bool store = !dry && l == p.L - 1 && p.write_y;
    int2* tab = nullptr;   // [T * k] (expert, gate bits)
    if (!rt && !dry && p.T * k <= 4096) {
        tab = reinterpret_cast<int2*>(scratch);
        for (int i = threadIdx.x; i < p.T * k; i += blockDim.x)
            tab[i] = make_int2(__ldcg(p.rb.idx + i), __float_as_int(__ldcg(p.rb.gate + i)));
        __syncthreads();
    }
    const int i0 = dry ? (int)threadIdx.x : blockIdx.x * blockDim.x + threadIdx.x;
    const int step = dry ? n : gridDim.x * blockDim.x;
    for (int i = i0; i < n; i += step) {
        const int t = i / H4, c4 = i % H4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < k; j0 += 8) {   // 8 slots' loads in flight, summed in slot order
            float g[8];
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = j0 + q;
                g[q] = 0.0f;
                v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < k) {
                    const int e = rt ? rt->idx[t * k + j] : tab ? tab[t * k + j].x : __ldcg(p.rb.idx + t * k + j);
                    if (e >= p.e_begin && e < p.e_end) {
                        g[q] = rt    ? rt->gate[t * k + j]
                               : tab ? __int_as_float(tab[t * k + j].y)
                                     : __ldcg(p.rb.gate + t * k + j);
                        v[q] = __ldcg(reinterpret_cast<const float4*>(p.ta.partial + (size_t)(t * k + j) * p.H) + c4);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (j0 + q < k && g[q] != 0.0f) {
                    acc.x = fmaf(g[q], v[q].x, acc.x);
                    acc.y = fmaf(g[q], v[q].y, acc.y);
                    acc.z = fmaf(g[q], v[q].z, acc.z);
                    acc.w = fmaf(g[q], v[q].w, acc.w);
                }
            }
        }
        if (store) {
            const size_t o = (size_t)t * p.H + (size_t)c4 * 4;
            if (p.y_bf16) {
                __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t*>(&a);
                u.y = *reinterpret_cast<uint32_t*>(&b);
                *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o) = u;
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o) = acc;
            }
        }
    }
}

// The expert phase of one layer, compiled as its own function (its register
// allocation does not carry the rest of the persistent kernel's live state).
template <bool kGathered, bool kNorm>
__device__ __noinline__ void persist_expert_phase(const TcArgs args, const TcMaps* maps, uint8_t* smem_raw,
                                                  uint32_t tmem, TcRoleState* rs, unsigned long long deadline) {
    using C = typename TcGeom<kGathered>::type;
    const TcSmem s = tc_smem<C>(smem_raw);
    if (threadIdx.x == C::kProducer * 32) {
        fence_proxy_async_global();   // inputs written by other CTAs before the last barrier / flag
        prefetch_tensormap(&maps->gate_q);
        prefetch_tensormap(&maps->up_q);
        prefetch_tensormap(&maps->down_q);
        prefetch_tensormap(&maps->gate_s);
        prefetch_tensormap(&maps->up_s);
        prefetch_tensormap(&maps->down_s);
    }
    TcRoleState r = *rs;
    tc_phase<C, kNorm>(*maps, args, s, tmem, r, deadline);
    *rs = r;
}

// This CTA's first router unit: its weight rows (and, for a plain input of one pass,
// its input rows) into shared memory, issued before anything else of the launch.
template <bool kLarge>
__device__ __forceinline__ void router_first_copies(const PersistParams& p, const TcSmem& sm, int* rstate) {
    if (p.norm) return;   // a residual stack has no router units (prep_unit forms the router products)
    if (p.rfull) {   // whole-row units: unit b on CTA b
        if ((int)blockIdx.x < router_full_units(p)) router_full_fetch(p, p.layer[0], blockIdx.x, sm);
        return;
    }
    const int units = router_units(p);
    if (threadIdx.x == 0) {
        rstate[2] = rstate[3] = -1;
        rstate[5] = rstate[6] = -1;   // no weight slice resident
        rstate[9] = 0;
    }
    const int u0 = router_first<kLarge>(units);
    if (u0 >= router_end<kLarge>(units)) return;
    router_fetch(p, p.layer[0], u0, sm);
    if (threadIdx.x == 0) {
        rstate[2] = u0;
        rstate[3] = 0;
    }
    if (!p.norm && p.T <= kPRouteTok && router_tblocks(p) == 1) {   // the pass's x rows, as router_unit copies them
        const int c0 = (u0 % (p.H / p.rslice)) * p.rslice;
        const int n16 = p.rslice / 8;
        const uint32_t xs_a = smem_u32(sm.slots), stride = router_stride(p);
        for (int i = threadIdx.x; i < p.T * n16; i += blockDim.x) {
            const int t = i / n16, c = (i % n16) * 8;
            cp_async_16(xs_a + (uint32_t)t * stride + (uint32_t)c * 2, p.x + (size_t)t * p.H + c0 + c);
        }
        if (threadIdx.x == 0) rstate[9] = 1;
    } else if (!p.norm && threadIdx.x < 32) {   // the first unit's input rows into L2
        const int lane = threadIdx.x;
        const int n_tb = router_tblocks(p);
        const int c0 = ((u0 / n_tb) % (p.H / p.rslice)) * p.rslice, tb0 = (u0 % n_tb) * p.rtok;
        for (int t = tb0 + lane; t < min(p.T, tb0 + min(p.rtok, 64)); t += 32)
            prefetch_l2(p.x + (size_t)t * p.H + c0, (uint32_t)p.rslice * 2);
    }
}

// All layers of one launch; returns early (in every thread of the block) on a timeout / abort.
// kLarge: the block is routed through the workspace (route_is_small(p) is false), with
// the input operand gathered per chunk; kNorm: a residual stack (p.norm).  The host
// launches the matching instantiation.
template <bool kLarge, bool kNorm>
__device__ __noinline__ void persist_layers(const PersistParams& p, uint8_t* smem_raw, uint32_t tmem,
                                            unsigned long long deadline) {
    using C = typename TcGeom<kLarge>::type;
    const TcSmem sm = tc_smem<C>(smem_raw);
    int* abort = p.wl.abort;
    int* status = p.ta.status;
    float* red = sm.red;                                   // block reductions (<= 32 floats)
    float* xs = reinterpret_cast<float*>(sm.slots);        // routing scratch
    unsigned btok = 0;   // thread 0: the grid-barrier word as this CTA's last arrival found it
    TcRoleState rs{0u, 0u, 0u, 0u};
    int* rstate = reinterpret_cast<int*>(sm.red + 40);     // router-weight copy state (router_fetch)
    const int units = p.rfull ? router_full_units(p) : router_units(p);
    const int cunits = p.T * (p.H / kCombineChunk);
    constexpr bool small = !kLarge;
    auto stamp = [&](int i) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[i] = globaltimer_ns();
    };
    float* ys = reinterpret_cast<float*>(sm.slots);        // prep_unit scratch (256 floats)
    stamp(0);   // (the first router unit's copies were issued before the setup)
    if constexpr (kNorm) {
        // residual stack: the first layer's inputs (its router products and operand); later
        // layers' inputs are prepared by the combine of the layer before
        for (int u = blockIdx.x; u < cunits; u += gridDim.x) stack_prep_unit(p, u, red, ys);
        grid_arrive(p.bar, btok, p.ta.debug_stall && blockIdx.x == gridDim.x - 1);
        // a CTA without a unit runs the routing code meanwhile (results discarded), so
        // that its code is in the caches when the grid needs it
        if (small && (int)blockIdx.x >= cunits) route_small(p, 0, reinterpret_cast<int*>(xs), sm.rt);
        if (!grid_wait(p.bar, btok, deadline, abort, status)) return;
    }
    stamp(1);

    for (int l = 0; l < p.L; ++l) {
        const PersistLayer& ly = p.layer[l];
        if constexpr (kNorm) {
            // (the inputs of this layer were prepared before the last grid barrier)
        } else if (p.rfull) {
            if ((int)blockIdx.x < units) router_full_unit(p, ly, blockIdx.x, sm);
        } else {
            for (int u = router_first<kLarge>(units); u < router_end<kLarge>(units); u += router_step<kLarge>())
                router_unit(p, ly, l, u, sm, rstate);
        }
        if constexpr (!kNorm) {
            if (threadIdx.x == 0) rstate[5] = -1;   // the slot area is reused from here on
            if (l == 0) stamp(53);
            // a CTA that ran a whole-row router unit holds x in shared memory
            operand_tasks(p, ly, p.rfull && (int)blockIdx.x < units ? sm.slots : nullptr);
            if (l == 0) stamp(54);
            const bool withhold = p.ta.debug_stall && l == 0 && blockIdx.x == gridDim.x - 1;
            grid_arrive(p.bar, btok, withhold);
            if (small && blockIdx.x >= units) {
                // a CTA without a router unit would only wait at the barrier: after arriving it
                // runs the routing code (results discarded; shared memory only) or, on every other
                // such CTA, the combine code (nothing stored), so that code is in L2 when the whole
                // grid needs it
                if (((blockIdx.x - units) & 1) == 0) route_small(p, l, reinterpret_cast<int*>(xs), sm.rt);
                else combine_elems(p, l, nullptr, sm.slots, true);
            }
            if (!grid_wait(p.bar, btok, deadline, abort, status)) return;
        }
        stamp(2 + 4 * l);
        if (small) {
            route_small(p, l, reinterpret_cast<int*>(xs), sm.rt);
            stamp(3 + 4 * l);
        } else {
            // larger blocks: top-k on every warp of the grid; grouping by CTA 0 while the
            // others wait on a release flag; the work list built by every CTA
            auto lstamp = [&](int i) {   // routing sub-steps of the first layer (CTA 0, profiling)
                if (l == 0) stamp(34 + i);
            };
            logits_reduce(p, ly);
            if (!grid_sync(p.bar, btok, deadline, abort, status)) return;
            lstamp(0);
            topk_tokens(p);
            if (!grid_sync(p.bar, btok, deadline, abort, status)) return;
            lstamp(1);
            if (blockIdx.x == 0) {
                route_phase(p, ly, l, reinterpret_cast<int*>(xs));
                __syncthreads();
                if (threadIdx.x == 0) {
                    __threadfence();
                    atomicExch(p.route_flag, l + 1);
                }
            } else {
                int failed = 0;
                if (threadIdx.x == 0) {
                    uint32_t spins = 0;
                    while (ld_acquire_gpu(p.route_flag) < l + 1) {
                        if ((++spins & 63u) == 0 && (globaltimer_ns() > deadline || aborted(abort))) {
                            failed = 1;
                            if (atomicExch(abort, 1) == 0) raise_status(status, MOE_ERR_TIMEOUT, -2);
                            break;
                        }
                    }
                }
                if (__syncthreads_or(failed)) return;
            }
            lstamp(2);
            build_items_slice(p, reinterpret_cast<int*>(xs));
            lstamp(3);
            gather_chunk_operand(p, reinterpret_cast<const int*>(xs), sm.slots);
            fence_proxy_async_global();   // read next by the expert phase's bulk copies
            lstamp(4);
            if (!grid_sync(p.bar, btok, deadline, abort, status)) return;
            stamp(3 + 4 * l);
        }
        if (kNorm && !small && threadIdx.x == 0) sm.rt->tscale_g = p.tscale;   // for the gate/up epilogue
        // the slots were written through the generic proxy; TMA writes them next
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        TcArgs ta = p.ta;
        ta.layer = p.layer_base + l;
        ta.queue = p.queues + l;
        ta.done = p.dones + (size_t)l * p.chunk_stride;
        ta.rt = small ? sm.rt : nullptr;
        if (l != 0 || p.layer_base != 0) ta.trace = nullptr;
        persist_expert_phase<kLarge, kNorm>(ta, &ly.maps, smem_raw, tmem, &rs, deadline);
        // the loader warps are done with the phase before the other roles (once the producer
        // has no more items): they run the combine code once without storing, so this SM's
        // instruction cache holds it when the combine starts after the barrier
        if (!kNorm && C::loader_index((int)(threadIdx.x >> 5)) >= 0)
            combine_elems(p, l, small ? sm.rt : nullptr, sm.slots, true);
        if (small && blockIdx.x == 0) publish_small(p, l, sm.rt);
        if (!grid_sync(p.bar, btok, deadline, abort, status)) return;
        stamp(4 + 4 * l);
        // the layer's expert phase is over in every CTA: its queue, done counters and the
        // routing flag go back to rest for the next launch (nothing reads them again here)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= p.chunk_stride; i += gridDim.x * blockDim.x) {
            if (i == 0) p.queues[l] = 0;
            else p.dones[(size_t)l * p.chunk_stride + i - 1] = 0;
        }
        if (!small && blockIdx.x == 0 && threadIdx.x == 0) *p.route_flag = 0;
        if constexpr (kNorm) {
            for (int u = blockIdx.x; u < cunits; u += gridDim.x)
                combine_unit(p, u, l, red, small ? sm.rt : nullptr, ys);
        } else {
            combine_elems(p, l, small ? sm.rt : nullptr, sm.slots);
        }
        stamp(5 + 4 * l);
        if (l + 1 < p.L) {
            grid_arrive(p.bar, btok);
            // a CTA without a combine unit runs the next layer's routing code meanwhile
            // (results discarded), so that its code is in the caches when the grid needs it
            if (small && (int)blockIdx.x >= cunits) route_small(p, l + 1, reinterpret_cast<int*>(xs), sm.rt);
            if (!grid_wait(p.bar, btok, deadline, abort, status)) return;
        }
    }
}

// The counters, flags and the grid-barrier word in the workspace are at rest (zero) when
// a launch starts and are returned to rest by the launch itself, so a forward issues no
// clearing copy before its kernel.  The host zeroes them once per workspace and writes
// the state tag beside them; a launch that finds another tag (the memory was used for
// something else since) records MOE_ERR_WORKSPACE and does nothing, and one that finds
// the abort flag of an earlier failed launch (its counters may not be at rest) does
// nothing either: the error stays in the status words until the host reads it and
// re-zeroes the state.
template <bool kLarge, bool kNorm>
__global__ void __launch_bounds__(kTcThreads, 1) persist_kernel(const __grid_constant__ PersistParams p) {
    extern __shared__ uint8_t smem_raw[];
    using C = typename TcGeom<kLarge>::type;
    const TcSmem sm = tc_smem<C>(smem_raw);
    // every thread reads the tag and the abort flag (nothing in this launch writes either
    // before its first grid barrier, so all threads see the same values); used after the setup
    const unsigned long long tag = *reinterpret_cast<const volatile unsigned long long*>(p.state_tag);
    const int aborted_before = *reinterpret_cast<const volatile int*>(p.wl.abort);
    router_first_copies<kLarge>(p, sm, reinterpret_cast<int*>(sm.red + 40));   // in flight during the setup
    const uint32_t tmem = tc_setup<C>(sm);
    const unsigned long long deadline = globaltimer_ns() + p.ta.timeout_ns;
    if (tag != p.tag) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            p.ta.status[0] = MOE_ERR_WORKSPACE;
            p.ta.status[1] = 0;
            *p.wl.abort = 1;
        }
    } else if (aborted_before == 0) {
        persist_layers<kLarge, kNorm>(p, smem_raw, tmem, deadline);
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.tstamp && blockIdx.x < 256)   // when each CTA finished (profiling)
        p.tstamp[56 + blockIdx.x] = globaltimer_ns();
    cp_async_wait_all();   // router-weight copies still in flight (a run cut short) land before exit
    tc_teardown<C>(sm, tmem, p.ta.timeout_ns);
}

}  // namespace moe
