// Persistent forward: one cooperative launch runs every phase of every layer
// ("MiMo 把 1T 模型推到每秒千 token", persistent engine kernel section: the whole
// pipeline stays resident instead of one launch per operator; implementation
// guide "关键实现细节" item 3: per-launch gaps of 5-10 us and 10-30% operator-boundary
// overhead at high token rates).  One CTA per SM, the expert kernel's block
// shape (16 warps) and tensor-memory allocation.  Per layer:
//   [router]           all CTAs, (32 experts x 1024 columns) units: partial logits
//                      and the layer input as the experts' E4M3-term operand
//   -- grid barrier --
//   [route]            small blocks (T*k <= 64): every CTA sums the slice partials
//                      (in order), takes the top-k and groups the pairs in its own
//                      shared memory (identical results everywhere; CTA 0 also
//                      publishes them); larger blocks: CTA 0 builds a global work
//                      list while the other CTAs wait on a release flag
//   [experts]          the work-queue expert phase of expert_tc.cuh
//   -- grid barrier --
//   [combine]          all CTAs, (token, 1024 columns) units: gate-weighted sum of
//                      the pair outputs, residual add, sums of squares for the next
//                      layer's RMSNorm
//   -- grid barrier --  (before the next layer's router)
// Every wait is bounded by the forward's deadline; a timeout sets the status
// word and the abort flag, and every CTA leaves at its next wait.
#pragma once

#include "expert_tc.cuh"
#include "route.cuh"

namespace moe {

constexpr int kMaxPersistLayers = 8;
constexpr int kPRouteExperts = 32;   // 16 warps x 2 expert rows
constexpr int kPRouteSlice = 1024;   // columns per router unit: 4 sub-chunks of 256 (8 per lane)
constexpr int kPRouteSub = 256;
constexpr int kPRouteTok = 8;        // tokens per round
constexpr int kCombineChunk = 1024;  // columns per combine unit

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
    float* ss;         // [T, ceil(H / 1024)] sums of squares of the residual per column chunk
    float* rpart;      // [H / 512, T, E]
    unsigned long long* tstamp;   // CTA 0's %globaltimer at phase ends (or NULL)
    TcArgs ta;         // expert phase: operands, partial, status, timeout (per-layer fields set per layer)
    RouteBufs rb;
    WorkList wl;       // items / n_items / abort for larger blocks
    int* queues;       // [kMaxPersistLayers] expert-phase queue per layer (zeroed per launch)
    int* dones;        // [kMaxPersistLayers, chunk_stride] finished gate/up items per chunk (zeroed per launch)
    int chunk_stride;
    unsigned* bar;     // grid barrier counter (zeroed per forward)
    int* route_flag;   // layers routed so far (zeroed per forward)
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

// All CTAs of the grid meet; bounded.  Returns false (in every thread) on timeout / abort.
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned& epoch, unsigned long long deadline,
                                          int* abort, int* status, bool withhold = false) {
    __syncthreads();
    ++epoch;
    int failed = 0;
    if (threadIdx.x == 0) {
        __threadfence();
        if (!withhold) atomicAdd(bar, 1u);
        const unsigned target = epoch * gridDim.x;
        uint32_t spins = 0;
        while (ld_acquire_u32(bar) < target) {
            if ((++spins & 63u) == 0 && (globaltimer_ns() > deadline || aborted(abort))) {
                failed = 1;
                if (atomicExch(abort, 1) == 0) raise_status(status, MOE_ERR_TIMEOUT, -1);
                break;
            }
        }
    }
    return __syncthreads_or(failed) == 0;
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

// 1/sqrt(mean(r^2) + eps) of token t from the chunk sums of squares (summed in
// chunk order by one warp: every caller gets the same value).
__device__ __forceinline__ float inv_rms(const PersistParams& p, int t) {
    const int lane = threadIdx.x & 31;
    const int nc = (p.H + kCombineChunk - 1) / kCombineChunk;
    float v = lane < nc ? __ldcg(p.ss + (size_t)t * nc + lane) : 0.0f;
    float tot = 0.0f;
    for (int c = 0; c < nc; ++c) tot += __shfl_sync(0xFFFFFFFFu, v, c);
    return 1.0f / sqrtf(tot / (float)p.H + p.eps);
}

// Router unit u = (expert group g of 32, column slice s of 1024): partial logits of
// the group over the slice for every token, 8 tokens at a time.  Each warp loads its
// 2 expert rows over the slice once; the slice of the layer input (x, or RMSNorm of
// the residual for a stack) is staged in shared memory once per token group; units
// of group 0 also write it as the expert phase's operand (8 E2M1 terms per block).
__device__ __noinline__ void router_unit(const PersistParams& p, const PersistLayer& ly, int u, float* xs /*[8][512]*/,
                                         float* sinv /*[8]*/) {
    const int H = p.H, E = p.E, T = p.T;
    const int n_sl = (H + kPRouteSlice - 1) / kPRouteSlice;
    const int eg = u / n_sl, sl = u % n_sl;
    const int c0 = sl * kPRouteSlice;
    const int ncols = min(kPRouteSlice, H - c0);   // 1024 or 512
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool computes = warp < 16;
    const int e0 = eg * kPRouteExperts + warp * 2;
    const int nsub = ncols / kPRouteSub;
    auto rs = [&](int i) {   // router timestamps of CTA 0's first unit (profiling)
        if (u == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[48 + i] = globaltimer_ns();
    };
    rs(0);
    // this warp's 2 expert rows over the slice, loaded once (8 bf16 per lane per sub-chunk)
    uint4 wreg[kPRouteSlice / kPRouteSub][2];
#pragma unroll
    for (int c = 0; c < kPRouteSlice / kPRouteSub; ++c)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int e = e0 + q;
            wreg[c][q] = (computes && e < E && c < nsub)
                             ? __ldg(reinterpret_cast<const uint4*>(ly.router_w + (size_t)e * H + c0 + c * kPRouteSub +
                                                                    lane * 8))
                             : make_uint4(0u, 0u, 0u, 0u);
        }
    for (int t0 = 0; t0 < T; t0 += kPRouteTok) {
        const int nt = min(kPRouteTok, T - t0);
        __syncthreads();
        if (t0 == 0) rs(1);
        if (p.norm && warp < nt) {
            const float v = inv_rms(p, t0 + warp);
            if (lane == 0) sinv[warp] = v;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nt * (ncols / 4); i += blockDim.x) {
            const int t = i / (ncols / 4), c = (i % (ncols / 4)) * 4;
            const size_t o = (size_t)(t0 + t) * H + c0 + c;
            float4 v;
            if (p.norm) {
                const float4 r = __ldcg(reinterpret_cast<const float4*>(p.resid + o));
                const uint2 wv = __ldg(reinterpret_cast<const uint2*>(ly.norm_w + c0 + c));
                const float iv = sinv[t];
                v = make_float4(r.x * iv * bf16_lo(wv.x), r.y * iv * bf16_hi(wv.x), r.z * iv * bf16_lo(wv.y),
                                r.w * iv * bf16_hi(wv.y));
            } else {
                const uint2 xv = __ldg(reinterpret_cast<const uint2*>(p.x + o));
                v = make_float4(bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y));
            }
            *reinterpret_cast<float4*>(xs + t * kPRouteSlice + c) = v;
        }
        __syncthreads();
        if (t0 == 0) rs(2);
        if (eg == 0) {
            // expert operand of this slice: 8 E2M1 terms per MX block (token, 32 columns)
            const int nb = ncols / 32;
            for (int i = warp; i < nt * nb; i += blockDim.x >> 5) {
                const int t = i / nb, kbl = i % nb;
                uint32_t sb0, sb1;
                const uint32_t codes = split_e2m1_terms(xs[t * kPRouteSlice + kbl * 32 + lane], sb0, sb1);
                store_act_terms(p.xb4, p.xsf, H, t0 + t, c0 / 32 + kbl, lane, codes, sb0, sb1);
            }
        }
        float accp[kPRouteTok][2];
#pragma unroll
        for (int t = 0; t < kPRouteTok; ++t)
#pragma unroll
            for (int q = 0; q < 2; ++q) accp[t][q] = 0.0f;
        if (computes) {
#pragma unroll
            for (int c = 0; c < kPRouteSlice / kPRouteSub; ++c) {
                if (c >= nsub) break;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float w[8];
                    const uint32_t* v = reinterpret_cast<const uint32_t*>(&wreg[c][q]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        w[2 * i] = bf16_lo(v[i]);
                        w[2 * i + 1] = bf16_hi(v[i]);
                    }
#pragma unroll
                    for (int t = 0; t < kPRouteTok; ++t) {
                        if (t < nt) {
                            const float4* xp =
                                reinterpret_cast<const float4*>(xs + t * kPRouteSlice + c * kPRouteSub + lane * 8);
                            const float4 xa = xp[0], xb = xp[1];
                            float a = accp[t][q];
                            a = fmaf(xa.x, w[0], a); a = fmaf(xa.y, w[1], a);
                            a = fmaf(xa.z, w[2], a); a = fmaf(xa.w, w[3], a);
                            a = fmaf(xb.x, w[4], a); a = fmaf(xb.y, w[5], a);
                            a = fmaf(xb.z, w[6], a); a = fmaf(xb.w, w[7], a);
                            accp[t][q] = a;
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kPRouteTok; ++t)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float v = warp_sum(accp[t][q]);
                    if (lane == q && t < nt && e0 + q < E) p.rpart[((size_t)sl * T + t0 + t) * E + e0 + q] = v;
                }
        }
        if (t0 == 0) rs(3);
    }
}

// Routing of a small verify block (T*k <= 64, T*E <= 8192) by every CTA into its own
// shared memory: logits from the slice partials (slice order), top-k + gates, and
// the grouping as a routing table for the expert phase.  All CTAs compute the same
// values; CTA 0 also publishes idx / gates / grouping for the combine and the
// debug copies.  scratch: >= T*E + 2*T*k + 2*E + 64 ints of shared memory.
__device__ __noinline__ void route_local(const PersistParams& p, const PersistLayer& ly, int l, int* scratch,
                                         RouteTable* rt) {
    const int T = p.T, E = p.E, k = p.k, H = p.H;
    const RouteBufs& rb = p.rb;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    auto sub = [&](int i) {   // sub-step timestamps of the first layer, CTA 0 (profiling)
        if (l == 0 && blockIdx.x == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[40 + i] = globaltimer_ns();
    };
    sub(0);
    float* lg = reinterpret_cast<float*>(scratch);   // [T * E]
    int* sidx = scratch + T * E;                     // [T * k]
    float* sgate = reinterpret_cast<float*>(sidx + T * k);
    int* cnt = sidx + 2 * T * k;                     // [E]
    int* fill = cnt + E;                             // [E]
    const int n_sl = (H + kPRouteSlice - 1) / kPRouteSlice;   // <= 16
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
        float a[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) a[q] = q < n_sl ? __ldcg(p.rpart + (size_t)q * T * E + i) : 0.0f;
        float z = 0.0f;
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (q < n_sl) z += a[q];
        lg[i] = z + (ly.router_b ? __ldg(ly.router_b + i % E) : 0.0f);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    sub(1);
    for (int t = warp; t < T; t += nw) {
        const float* lrow = lg + (size_t)t * E;
        float lv[kMaxExperts / 32];
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane + 32 * i;
            float v = e < E ? lrow[e] : __int_as_float(0xFF800000);
            if (v != v) v = __int_as_float(0xFF800000);
            lv[i] = v;
        }
        float prev_v = __int_as_float(0x7F800000);
        int prev_e = -1;
        float my_sel = 0.0f;
        for (int j = 0; j < k; ++j) {
            float bv = __int_as_float(0xFF800000);
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; ++i) {
                const int e = lane + 32 * i;
                if (e < E && route_before(prev_v, prev_e, lv[i], e) && route_before(lv[i], e, bv, be)) {
                    bv = lv[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
                if (route_before(ov, oe, bv, be)) { bv = ov; be = oe; }
            }
            prev_v = bv;
            prev_e = be;
            if (lane == j) my_sel = bv;
            if (lane == 0) sidx[t * k + j] = be;
        }
        const float m = __shfl_sync(0xFFFFFFFFu, my_sel, 0);
        const float ex = lane < k ? expf(my_sel - m) : 0.0f;
        const float den = warp_sum(ex);
        if (lane < k) sgate[t * k + lane] = ex / den;
    }
    __syncthreads();
    sub(2);
    const int npairs = T * k;
    if (warp == 0) {
        // counts -> offsets (scan over E) and the routed experts in ascending id
        for (int s = lane; s < npairs; s += 32) {
            const int e = sidx[s];
            if (e >= p.e_begin && e < p.e_end) atomicAdd(&cnt[e], 1);
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) fill[e] = cnt[e] > 0 ? 1 : 0;
        __syncwarp();
        const int n_active = warp_excl_scan(fill, E);   // fill -> position among the routed experts
        __syncwarp();
        for (int e = lane; e < E; e += 32)
            if (cnt[e] > 0) rt->e[fill[e]] = e;
        __syncwarp();
        // per routed expert: first perm position (its pairs in (t, j) order) and chunks
        int run = 0, chunks = 0;
        for (int a0 = 0; a0 < n_active; a0 += 32) {
            const int a = a0 + lane;
            const int c = a < n_active ? cnt[rt->e[a]] : 0;
            const int ch = (c + kTmaTok - 1) / kTmaTok;
            int ic = c, ich = ch;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, ic, o);
                const int v = __shfl_up_sync(0xFFFFFFFFu, ich, o);
                if (lane >= o) { ic += u; ich += v; }
            }
            if (a < n_active) {
                rt->beg[a] = run + ic - c;
                rt->cnt[a] = c;
                rt->chunk0[a] = chunks + ich - ch;
                fill[rt->e[a]] = run + ic - c;   // running fill position of the expert
            }
            run += __shfl_sync(0xFFFFFFFFu, ic, 31);
            chunks += __shfl_sync(0xFFFFFFFFu, ich, 31);
        }
        __syncwarp();
        if (lane == 0) {
            rt->n_active = n_active;
            rt->n_chunks = chunks;
            rt->pad0 = run;   // pairs routed into the shard
            for (int s = 0; s < npairs; ++s) {   // pairs in (t, j) order
                const int e = sidx[s];
                if (e < p.e_begin || e >= p.e_end) continue;
                const int pos = fill[e]++;
                rt->tok[pos] = s / k;
                rt->pair[pos] = s;
            }
        }
    }
    __syncthreads();
    sub(3);
    if (blockIdx.x == 0) {   // publish for the combine, the down epilogue's caller and the debug copies
        for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
            rb.idx[i] = sidx[i];
            rb.gate[i] = sgate[i];
        }
        for (int i = threadIdx.x; i < T * E; i += blockDim.x) rb.logits[i] = lg[i];
        const int na = rt->n_active;
        for (int e = threadIdx.x; e < E; e += blockDim.x) rb.counts[e] = cnt[e];
        for (int i = threadIdx.x; i < npairs; i += blockDim.x) rb.perm[i] = i < rt->pad0 ? rt->pair[i] : -1;
        for (int a = threadIdx.x; a < na; a += blockDim.x) rb.active[1 + a] = rt->e[a];
        if (threadIdx.x == 0) rb.active[0] = na;
        __syncthreads();
        // offsets: exclusive prefix of counts
        if (warp == 0) {
            for (int e = lane; e < E; e += 32) fill[e] = cnt[e];
            __syncwarp();
            const int total = warp_excl_scan(fill, E);
            __syncwarp();
            for (int e = lane; e <= E; e += 32) rb.offsets[e] = e < E ? fill[e] : total;
        }
        __syncthreads();
        const int lgi = p.layer_base + l;
        if (p.dbg.idx) for (int i = threadIdx.x; i < npairs; i += blockDim.x) p.dbg.idx[(size_t)lgi * npairs + i] = sidx[i];
        if (p.dbg.gate) for (int i = threadIdx.x; i < npairs; i += blockDim.x) p.dbg.gate[(size_t)lgi * npairs + i] = sgate[i];
        if (p.dbg.perm) for (int i = threadIdx.x; i < npairs; i += blockDim.x) p.dbg.perm[(size_t)lgi * npairs + i] = rb.perm[i];
        if (p.dbg.counts) for (int i = threadIdx.x; i < E; i += blockDim.x) p.dbg.counts[(size_t)lgi * E + i] = cnt[i];
        if (p.dbg.offsets)
            for (int i = threadIdx.x; i <= E; i += blockDim.x) p.dbg.offsets[(size_t)lgi * (E + 1) + i] = rb.offsets[i];
    }
    sub(4);
}

// Combine unit (token t, column chunk c of 1024): out = sum_j gate[t, j] *
// partial[t*k + j] (slots in order, pairs outside the expert shard skipped); with a
// residual stack r += out and the chunk's sum of squares of r is kept for the next
// RMSNorm.  The last layer writes y.
__device__ __noinline__ void combine_unit(const PersistParams& p, int u, int l, float* red) {
    const int H = p.H, k = p.k;
    const int nc = (H + kCombineChunk - 1) / kCombineChunk;
    const int t = u / nc, c = u % nc;
    const int c0 = c * kCombineChunk, ncols = min(kCombineChunk, H - c0);
    const RouteBufs& rb = p.rb;
    const bool last = l == p.L - 1;
    const size_t o = (size_t)t * H + c0;
    float gj[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {   // gates of the slots in the shard (0 outside)
        gj[j] = 0.0f;
        if (j < k) {
            const int e = __ldcg(rb.idx + t * k + j);
            gj[j] = (e >= p.e_begin && e < p.e_end) ? __ldcg(rb.gate + t * k + j) : 0.0f;
        }
    }
    float ssl = 0.0f;
    const int h = threadIdx.x * 4;
    if (h < ncols) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j >= k || gj[j] == 0.0f) continue;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ta.partial + (size_t)(t * k + j) * H + c0 + h));
            acc.x = fmaf(gj[j], v.x, acc.x);
            acc.y = fmaf(gj[j], v.y, acc.y);
            acc.z = fmaf(gj[j], v.z, acc.z);
            acc.w = fmaf(gj[j], v.w, acc.w);
        }
        if (p.norm) {
            const float4 r = __ldcg(reinterpret_cast<const float4*>(p.resid + o + h));
            acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
            *reinterpret_cast<float4*>(p.resid + o + h) = acc;
            ssl = acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
        }
        if (last && p.write_y) {
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
        if (threadIdx.x == 0) p.ss[(size_t)t * nc + c] = tot;
    }
}

// Residual start of a stack, unit (token t, chunk c): r = fp32(x) and the chunk's sum of squares.
__device__ __noinline__ void stack_init_unit(const PersistParams& p, int u, float* red) {
    const int H = p.H;
    const int nc = (H + kCombineChunk - 1) / kCombineChunk;
    const int t = u / nc, c = u % nc;
    const int c0 = c * kCombineChunk, ncols = min(kCombineChunk, H - c0);
    const size_t o = (size_t)t * H + c0;
    float ssl = 0.0f;
    const int h = threadIdx.x * 4;
    if (h < ncols) {
        const uint2 xv = __ldg(reinterpret_cast<const uint2*>(p.x + o + h));
        const float4 v = make_float4(bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y));
        *reinterpret_cast<float4*>(p.resid + o + h) = v;
        ssl = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    const float tot = block_sum(ssl, red);
    if (threadIdx.x == 0) p.ss[(size_t)t * nc + c] = tot;
}


// Routing of one layer by one block: logits from the slice partials (fixed order),
// top-k + gates, grouping (counts, offsets, perm, active list) and the work list.
// scratch: shared memory of at least (2 * E + 1 + 32 * E + 64) ints.
__device__ __noinline__ void route_phase(const PersistParams& p, const PersistLayer& ly, int l, int* scratch) {
    const int T = p.T, E = p.E, k = p.k, H = p.H;
    const RouteBufs& rb = p.rb;
    const WorkList& wl = p.wl;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    auto sub = [&](int i) {   // sub-step timestamps of the first layer (profiling)
        if (l == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[40 + i] = globaltimer_ns();
    };
    sub(0);
    // ---- logits: the slice partials summed in slice order; all slices of an
    // element are loaded together (H / 512 <= 32)
    const int n_sl = (H + kPRouteSlice - 1) / kPRouteSlice;   // <= 16
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
        float a[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) a[q] = q < n_sl ? __ldcg(p.rpart + (size_t)q * T * E + i) : 0.0f;
        float z = 0.0f;
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (q < n_sl) z += a[q];
        rb.logits[i] = z + (ly.router_b ? ly.router_b[i % E] : 0.0f);
    }
    __syncthreads();
    // ---- top-k + gates, one warp per token (logits of lane l: experts l, l+32, ...)
    for (int t = warp; t < T; t += nw) {
        const float* lrow = rb.logits + (size_t)t * E;
        float lv[kMaxExperts / 32];
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane + 32 * i;
            float v = e < E ? __ldcg(lrow + e) : __int_as_float(0xFF800000);
            if (v != v) v = __int_as_float(0xFF800000);
            lv[i] = v;
        }
        float prev_v = __int_as_float(0x7F800000);
        int prev_e = -1;
        float my_sel = 0.0f;
        for (int j = 0; j < k; ++j) {
            float bv = __int_as_float(0xFF800000);
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; ++i) {
                const int e = lane + 32 * i;
                if (e < E && route_before(prev_v, prev_e, lv[i], e) && route_before(lv[i], e, bv, be)) {
                    bv = lv[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
                if (route_before(ov, oe, bv, be)) { bv = ov; be = oe; }
            }
            prev_v = bv;
            prev_e = be;
            if (lane == j) my_sel = bv;
            if (lane == 0) rb.idx[t * k + j] = be;
        }
        const float m = __shfl_sync(0xFFFFFFFFu, my_sel, 0);
        const float ex = lane < k ? expf(my_sel - m) : 0.0f;
        const float den = warp_sum(ex);
        if (lane < k) rb.gate[t * k + lane] = ex / den;
    }
    sub(1);
    int* cnt = scratch;                  // [E]
    int* flag = scratch + E;             // [E + 1]
    int* wcnt = scratch + 2 * E + 1;     // [32][E] (nw <= 32)
    int* misc = wcnt + 32 * E;           // [64]
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int npairs = T * k;
    for (int s = threadIdx.x; s < npairs; s += blockDim.x) {
        const int e = rb.idx[s];
        if (e >= p.e_begin && e < p.e_end) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    sub(2);
    // ---- counts, offsets, active list (warp 0)
    if (warp == 0) {
        for (int e = lane; e < E; e += 32) {
            rb.counts[e] = cnt[e];
            flag[e] = cnt[e] > 0 ? 1 : 0;
        }
        __syncwarp();
        const int total = warp_excl_scan(cnt, E);            // cnt -> offsets
        __syncwarp();
        const int n_active = warp_excl_scan(flag, E);        // flag -> active position
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            rb.offsets[e] = cnt[e];
            if (rb.counts[e] > 0) rb.active[1 + flag[e]] = e;
        }
        if (lane == 0) {
            rb.offsets[E] = total;
            rb.active[0] = n_active;
            misc[0] = n_active;
        }
    }
    __syncthreads();
    // ---- perm: pairs in id order inside each expert (rounds of blockDim pairs)
    for (int base = 0; base < npairs; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int e = -1;
        if (s < npairs) {
            e = rb.idx[s];
            if (e < p.e_begin || e >= p.e_end) e = -1;
        }
        for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const int lane_rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && lane_rank == 0) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int run = cnt[x];
            for (int w = 0; w < nw; ++w) {
                const int c = wcnt[w * E + x];
                wcnt[w * E + x] = run;
                run += c;
            }
            cnt[x] = run;
        }
        __syncthreads();
        if (e >= 0) rb.perm[wcnt[warp * E + e] + lane_rank] = s;
        __syncthreads();
    }
    sub(3);
    // ---- work list: chunks of <= 8 pairs per routed expert.  The grouping is
    // staged in shared memory first (the item records read it many times).
    const int n_active = misc[0];
    const int rbu = p.I / kTmaRows, rbd = H / kDownRows;
    int* chunk0 = flag;                 // [n_active]: first chunk index of each routed expert
    int* s_act = wcnt;                  // [n_active] expert ids
    int* s_beg = wcnt + E;              // [n_active] first perm position
    int* s_cnt = wcnt + 2 * E;          // [n_active] pairs
    int* s_perm = wcnt + 3 * E;         // [T * k] pair id of each perm position
    for (int a = threadIdx.x; a < n_active; a += blockDim.x) {
        const int e = __ldcg(rb.active + 1 + a);
        s_act[a] = e;
        s_beg[a] = __ldcg(rb.offsets + e);
        s_cnt[a] = __ldcg(rb.counts + e);
    }
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) s_perm[i] = __ldcg(rb.perm + i);
    __syncthreads();
    if (warp == 0) {
        for (int a = lane; a < n_active; a += 32) {
            chunk0[a] = (s_cnt[a] + kTmaTok - 1) / kTmaTok;
        }
        __syncwarp();
        const int total_chunks = warp_excl_scan(chunk0, n_active);
        if (lane == 0) {
            misc[1] = total_chunks;
            wl.n_items[0] = total_chunks * (rbu + rbd);
            wl.n_items[1] = total_chunks * rbu;
        }
    }
    __syncthreads();
    const int total_chunks = misc[1];
    const int n_gu = total_chunks * rbu;
    for (int i = threadIdx.x; i < total_chunks * (rbu + rbd); i += blockDim.x) {
        const bool down = i >= n_gu;
        const int j = down ? i - n_gu : i;
        const int nrb = down ? rbd : rbu;
        const int chunk = j / nrb, rbi = j % nrb;
        int lo = 0, hi = n_active - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk0[mid] <= chunk) lo = mid; else hi = mid - 1;
        }
        const int tc = chunk - chunk0[lo];
        ItemRec r;
        r.code = item_code(down ? kItemDown : kItemGateUp, rbi, tc, lo);
        r.e = s_act[lo];
        r.beg = s_beg[lo] + tc * kTmaTok;
        r.ntok = min(kTmaTok, s_cnt[lo] - tc * kTmaTok);
#pragma unroll
        for (int q = 0; q < kTmaTok; ++q) r.tok[q] = q < r.ntok ? (down ? s_perm[r.beg + q] : s_perm[r.beg + q] / k) : 0;
        r.chunk = chunk;
#pragma unroll
        for (int q = 0; q < 3; ++q) r.pad[q] = 0;
        wl.items[i] = r;
    }
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

// The expert phase of one layer, compiled as its own function (its register
// allocation does not carry the rest of the persistent kernel's live state).
__device__ __noinline__ void persist_expert_phase(const TcArgs args, const TcMaps* maps, uint8_t* smem_raw,
                                                  uint32_t tmem, TcRoleState* rs, unsigned long long deadline) {
    const TcSmem s = tc_smem(smem_raw);
    if (threadIdx.x == kTcWarpProducer * 32) {
        fence_proxy_async_global();   // inputs written by other CTAs before the last barrier / flag
        prefetch_tensormap(&maps->gate_q);
        prefetch_tensormap(&maps->up_q);
        prefetch_tensormap(&maps->down_q);
        prefetch_tensormap(&maps->gate_s);
        prefetch_tensormap(&maps->up_s);
        prefetch_tensormap(&maps->down_s);
    }
    TcRoleState r = *rs;
    tc_phase(*maps, args, s, tmem, r, deadline);
    *rs = r;
}

// All layers of one launch; returns early (in every thread of the block) on a timeout / abort.
__device__ __noinline__ void persist_layers(const PersistParams& p, uint8_t* smem_raw, uint32_t tmem,
                                            unsigned long long deadline) {
    const TcSmem sm = tc_smem(smem_raw);
    int* abort = p.wl.abort;
    int* status = p.ta.status;
    float* red = sm.red;                                   // block reductions (<= 32 floats)
    float* xs = reinterpret_cast<float*>(sm.slots);        // router staging / routing scratch
    float* sinv = sm.red + 32;                             // [8]
    unsigned epoch = 0;
    TcRoleState rs{0u, 0u, 0u, 0u};
    const int n_sl = (p.H + kPRouteSlice - 1) / kPRouteSlice;
    const int units = ((p.E + kPRouteExperts - 1) / kPRouteExperts) * n_sl;
    const int cunits = p.T * ((p.H + kCombineChunk - 1) / kCombineChunk);
    const bool small = p.T * p.k <= kRtMaxPairs && p.T * p.E <= 8192;
    auto stamp = [&](int i) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && p.tstamp) p.tstamp[i] = globaltimer_ns();
    };
    stamp(0);
    if (p.norm && p.init_from_x) {
        for (int u = blockIdx.x; u < cunits; u += gridDim.x) stack_init_unit(p, u, red);
        if (!grid_sync(p.bar, epoch, deadline, abort, status)) return;
    }
    stamp(1);

    for (int l = 0; l < p.L; ++l) {
        const PersistLayer& ly = p.layer[l];
        for (int u = blockIdx.x; u < units; u += gridDim.x) router_unit(p, ly, u, xs, sinv);
        const bool withhold = p.ta.debug_stall && l == 0 && blockIdx.x == gridDim.x - 1;
        if (!grid_sync(p.bar, epoch, deadline, abort, status, withhold)) return;
        stamp(2 + 4 * l);
        if (small) {
            route_local(p, ly, l, reinterpret_cast<int*>(xs), sm.rt);
            __syncthreads();
            stamp(3 + 4 * l);
        } else if (blockIdx.x == 0) {
            route_phase(p, ly, l, reinterpret_cast<int*>(xs));
            __syncthreads();
            stamp(3 + 4 * l);
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
        // the slots were written through the generic proxy; TMA writes them next
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        TcArgs ta = p.ta;
        ta.layer = p.layer_base + l;
        ta.queue = p.queues + l;
        ta.done = p.dones + (size_t)l * p.chunk_stride;
        ta.rt = small ? sm.rt : nullptr;
        if (l != 0 || p.layer_base != 0) ta.trace = nullptr;
        persist_expert_phase(ta, &ly.maps, smem_raw, tmem, &rs, deadline);
        if (!grid_sync(p.bar, epoch, deadline, abort, status)) return;
        stamp(4 + 4 * l);
        for (int u = blockIdx.x; u < cunits; u += gridDim.x) combine_unit(p, u, l, red);
        stamp(5 + 4 * l);
        if (l + 1 < p.L && !grid_sync(p.bar, epoch, deadline, abort, status)) return;
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) persist_kernel(const __grid_constant__ PersistParams p) {
    extern __shared__ uint8_t smem_raw[];
    const TcSmem sm = tc_smem(smem_raw);
    const uint32_t tmem = tc_setup(sm);
    const unsigned long long deadline = globaltimer_ns() + p.ta.timeout_ns;
    persist_layers(p, smem_raw, tmem, deadline);
    tc_teardown(sm, tmem, p.ta.timeout_ns);
}

}  // namespace moe
