// Routing phase of one MoE layer: router GEMM, top-k + softmax gates, and the
// token-to-expert grouping (counts, offsets, perm, active expert list).
//
// The router stays in higher precision than the experts ("MiMo x TileRT",
// section "第一层：FP4 选择性量化"; "MiMo 把 1T 模型推到每秒千 token", section
// "FP4：只量化 MoE expert": the router's top-k choice is precision-sensitive),
// so logits are accumulated in fp32 from bf16 weights and fp32 activations, in
// a fixed order (deterministic).
#pragma once

#include "common.cuh"

namespace moe {

// logits[t, e] = sum_h act[t, h] * Wr[e, h] + b[e].
// One warp per expert row; the row is read once in 16-byte vectors and applied
// to up to 8 tokens at a time.  Grid: ceil(E / warps_per_block) blocks.
__global__ void __launch_bounds__(256) route_logits_kernel(const float* __restrict__ act, int T, int H,
                                                           const __nv_bfloat16* __restrict__ wr,
                                                           const float* __restrict__ bias, int E,
                                                           float* __restrict__ logits) {
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (e >= E) return;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    const int nvec = H / 8;
    const float b = bias ? bias[e] : 0.0f;
    for (int t0 = 0; t0 < T; t0 += 8) {
        const int nt = min(8, T - t0);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int c = lane; c < nvec; c += 32) {
            const uint4 wv = __ldg(wrow + c);
            const float w[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                                bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < nt) {
                    const float4* xp = reinterpret_cast<const float4*>(act + (size_t)(t0 + i) * H) + 2 * c;
                    const float4 a0 = __ldg(xp), a1 = __ldg(xp + 1);
                    float s = acc[i];
                    s = fmaf(a0.x, w[0], s); s = fmaf(a0.y, w[1], s);
                    s = fmaf(a0.z, w[2], s); s = fmaf(a0.w, w[3], s);
                    s = fmaf(a1.x, w[4], s); s = fmaf(a1.y, w[5], s);
                    s = fmaf(a1.z, w[6], s); s = fmaf(a1.w, w[7], s);
                    acc[i] = s;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float s = warp_sum(acc[i]);
            if (lane == 0 && i < nt) logits[(size_t)(t0 + i) * E + e] = s + b;
        }
    }
}

// Partial router logits over 512-column slices of H:
//   partial[s, t, e] = sum_{h in slice s} act[t, h] * Wr[e, h].
// Grid (ceil(E / 32), H / 512), 256 threads.  Each warp owns 4 expert rows and
// keeps their 512-column slice in registers (lane l: columns 16l..16l+15); the
// block stages the activations of 16 tokens at a time in shared memory, so each
// weight byte and each activation byte is read once.  The slices are summed in
// a fixed order by route_select_kernel (deterministic).
constexpr int kRouteSlice = 512;
constexpr int kRouteTokGroup = 16;
__global__ void __launch_bounds__(256) route_partial_kernel(const float* __restrict__ act, int T, int H,
                                                            const __nv_bfloat16* __restrict__ wr, int E,
                                                            float* __restrict__ partial) {
    __shared__ __align__(16) float xs[kRouteTokGroup][kRouteSlice];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slice = blockIdx.y;
    const int c0 = slice * kRouteSlice + lane * 16;
    const int e0 = blockIdx.x * 32 + warp * 4;
    float w[4][16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int e = e0 + q;
        if (e < E) {
            const uint4* src = reinterpret_cast<const uint4*>(wr + (size_t)e * H + c0);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                w[q][2 * i] = bf16_lo(v[i]);
                w[q][2 * i + 1] = bf16_hi(v[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[q][i] = 0.0f;
        }
    }
    for (int t0 = 0; t0 < T; t0 += kRouteTokGroup) {
        const int nt = min(kRouteTokGroup, T - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * (kRouteSlice / 4); i += blockDim.x) {
            const int t = i / (kRouteSlice / 4), c = i % (kRouteSlice / 4);
            reinterpret_cast<float4*>(xs[t])[c] =
                __ldg(reinterpret_cast<const float4*>(act + (size_t)(t0 + t) * H + slice * kRouteSlice) + c);
        }
        __syncthreads();
        for (int t = 0; t < nt; ++t) {
            const float4* xp = reinterpret_cast<const float4*>(&xs[t][lane * 16]);
            float x[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = xp[i];
                x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float acc = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc = fmaf(x[i], w[q][i], acc);
                acc = warp_sum(acc);
                if (lane == q && e0 + q < E) partial[((size_t)slice * T + t0 + t) * E + e0 + q] = acc;
            }
        }
    }
}

// (v1, e1) comes before (v2, e2) in routing order: larger logit first, then lower index.
__device__ __forceinline__ bool route_before(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
// scratch: 33 ints; the total lands in scratch[32].
__device__ __forceinline__ int block_excl_scan_1024(int v, int* scratch) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int s = scratch[lane];
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, si, o);
            if (lane >= o) si += n;
        }
        scratch[lane] = si - s;  // exclusive prefix of the warp totals
        if (lane == 31) scratch[32] = si;
    }
    __syncthreads();
    const int r = scratch[w] + incl - v;
    __syncthreads();
    return r;
}

// Top-k, softmax gates and the grouping of (token, slot) pairs by expert.
// One block of 1024 threads.  Pairs routed outside [e_begin, e_end) are not
// grouped (another shard computes them).  Dynamic shared memory:
// (33 * E + 64) ints.
__global__ void __launch_bounds__(1024) route_select_kernel(const float* logits, int T, int E, int k,
                                                            int e_begin, int e_end, RouteBufs rb,
                                                            const float* __restrict__ partial = nullptr,
                                                            int n_slices = 0, const float* __restrict__ bias = nullptr) {
    extern __shared__ int smem[];
    if (partial) {
        // logits = bias + sum of the slice partials, slices in ascending order
        for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
            float z = 0.0f;
            for (int s0 = 0; s0 < n_slices; s0 += 16) {   // up to 16 independent loads in flight
                float a[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) a[u] = s0 + u < n_slices ? partial[(size_t)(s0 + u) * T * E + i] : 0.0f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (s0 + u < n_slices) z += a[u];
            }
            rb.logits[i] = z + (bias ? bias[i % E] : 0.0f);
        }
        __syncthreads();
        logits = rb.logits;
    }
    int* cnt = smem;                 // [E]
    int* wcnt = smem + E;            // [32][E] per-warp counts, then their running prefix
    int* scratch = wcnt + 32 * E;    // [64]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // ---- top-k + gates: one warp per token, k rounds of a warp arg-max that
    // only admits candidates after the previous pick in routing order.  Lane l
    // keeps the logits of experts l, l+32, ... in registers (E <= 1024).
    for (int t = warp; t < T; t += 32) {
        const float* lrow = logits + (size_t)t * E;
        float lv[kMaxExperts / 32];
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane + 32 * i;
            float v = e < E ? lrow[e] : __int_as_float(0xFF800000);
            if (v != v) v = __int_as_float(0xFF800000);  // NaN ranks last
            lv[i] = v;
        }
        float prev_v = __int_as_float(0x7F800000);  // +inf
        int prev_e = -1;
        float my_sel = 0.0f;
        for (int j = 0; j < k; ++j) {
            float bv = __int_as_float(0xFF800000);  // -inf
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; ++i) {
                const int e = lane + 32 * i;
                const float v = lv[i];
                if (e < E && route_before(prev_v, prev_e, v, e) && route_before(v, e, bv, be)) { bv = v; be = e; }
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
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();

    // ---- counts
    const int npairs = T * k;
    for (int s = threadIdx.x; s < npairs; s += blockDim.x) {
        const int e = rb.idx[s];
        if (e >= e_begin && e < e_end) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();

    // ---- offsets (exclusive scan of counts) and the active expert list
    {
        const int e = threadIdx.x;
        const int c = e < E ? cnt[e] : 0;
        const int off = block_excl_scan_1024(c, scratch);
        if (e < E) rb.offsets[e] = off;
        if (e == 0) rb.offsets[E] = scratch[32];
        if (e < E) rb.counts[e] = c;
        const int flag = (e < E && c > 0) ? 1 : 0;
        const int pos = block_excl_scan_1024(flag, scratch);
        if (flag) rb.active[1 + pos] = e;
        if (e == 0) rb.active[0] = scratch[32];
        if (e < E) cnt[e] = off;  // running base of each expert's list
    }
    __syncthreads();

    // ---- perm: pairs in ascending id order inside each expert.  Pairs are
    // taken in rounds of 1024 (id order); inside a round a pair's rank is the
    // number of same-expert pairs before it: earlier warps via the per-warp
    // count prefix, earlier lanes via a match mask.
    for (int base = 0; base < npairs; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int e = -1;
        if (s < npairs) {
            e = rb.idx[s];
            if (e < e_begin || e >= e_end) e = -1;
        }
        for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
        const int lane_rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && lane_rank == 0) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int run = cnt[x];
            for (int w = 0; w < 32; ++w) {
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
}

}  // namespace moe
