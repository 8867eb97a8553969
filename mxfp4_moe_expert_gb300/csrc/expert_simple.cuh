// Multi-kernel comparison path of the expert FFN: one launch per phase, plain
// coalesced 16-byte loads, fp32 dequant + FMA.
//
// Expert FFN (implementation guide, "关键实现细节" item 1: gate_proj / up_proj /
// down_proj; SwiGLU activation): a = silu(Wg x) * (Wu x), d = Wd a.  Weights are
// MXFP4: element c of row r = e2m1(nibble) * 2^(S[r, c/32] - 127) (OCP MX v1.0).
#pragma once

#include "common.cuh"

namespace moe {

struct ExpertWeights {
    const uint8_t* gate_q;
    const uint8_t* gate_s;
    const uint8_t* up_q;
    const uint8_t* up_s;
    const uint8_t* down_q;
    const uint8_t* down_s;
};

// Decodes the 32 E2M1 codes of a 16-byte vector and returns sum_c w_c * x_c
// (unscaled: the caller multiplies by the block scale).
__device__ __forceinline__ float dot32_e2m1(const uint4 q, const float* __restrict__ x) {
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
    const float4* xp = reinterpret_cast<const float4*>(x);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 a = __ldg(xp + 2 * i), b = __ldg(xp + 2 * i + 1);
        const uint32_t w = wv[i];
        s = fmaf(e2m1_to_f32(w), a.x, s);
        s = fmaf(e2m1_to_f32(w >> 4), a.y, s);
        s = fmaf(e2m1_to_f32(w >> 8), a.z, s);
        s = fmaf(e2m1_to_f32(w >> 12), a.w, s);
        s = fmaf(e2m1_to_f32(w >> 16), b.x, s);
        s = fmaf(e2m1_to_f32(w >> 20), b.y, s);
        s = fmaf(e2m1_to_f32(w >> 24), b.z, s);
        s = fmaf(e2m1_to_f32(w >> 28), b.w, s);
    }
    return s;
}

// h[p, r] = silu(Wg_e[r] . act[t_p]) * (Wu_e[r] . act[t_p]) for every pair p of
// every routed expert e (p = position in perm).  Grid (I / 32, max_active),
// 256 threads: each warp owns 4 rows; lanes split the contraction.
__global__ void __launch_bounds__(256) gateup_simple_kernel(const float* __restrict__ act, int H, int I, int k,
                                                           ExpertWeights w, RouteBufs rb, float* __restrict__ hbuf,
                                                           int* status, int layer) {
    const int a = blockIdx.y;
    if (a >= rb.active[0]) return;
    const int e = rb.active[1 + a];
    const int beg = rb.offsets[e], n = rb.counts[e];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nblk = H / kMxBlock;
    for (int rr = 0; rr < 4; ++rr) {
        const int r = blockIdx.x * 32 + warp * 4 + rr;
        const size_t row = (size_t)e * I + r;
        const uint4* gq = reinterpret_cast<const uint4*>(w.gate_q + row * (H / 2));
        const uint4* uq = reinterpret_cast<const uint4*>(w.up_q + row * (H / 2));
        const uint8_t* gs = w.gate_s + row * nblk;
        const uint8_t* us = w.up_s + row * nblk;
        for (int i0 = 0; i0 < n; i0 += 8) {
            const int ni = min(8, n - i0);
            int tok[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) tok[i] = i < ni ? rb.perm[beg + i0 + i] / k : 0;
            float ag[8], au[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) { ag[i] = 0.0f; au[i] = 0.0f; }
            for (int blk = lane; blk < nblk; blk += 32) {
                const uint4 qg = __ldg(gq + blk), qu = __ldg(uq + blk);
                const uint32_t sgb = gs[blk], sub = us[blk];
                if (sgb == 0xFFu || sub == 0xFFu) raise_status(status, MOE_ERR_BAD_SCALE, layer * 65536 + e);
                const float sg = e8m0_to_f32(sgb), su = e8m0_to_f32(sub);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i < ni) {
                        const float* x = act + (size_t)tok[i] * H + blk * kMxBlock;
                        ag[i] = fmaf(dot32_e2m1(qg, x), sg, ag[i]);
                        au[i] = fmaf(dot32_e2m1(qu, x), su, au[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float g = warp_sum(ag[i]);
                const float u = warp_sum(au[i]);
                if (lane == 0 && i < ni) hbuf[(size_t)(beg + i0 + i) * I + r] = silu(g) * u;
            }
        }
    }
}

// partial[s, r] = Wd_e[r] . h[p] for every pair p (pair id s = perm[p]) of every
// routed expert.  Grid (H / 32, max_active), 256 threads, as above.
__global__ void __launch_bounds__(256) down_simple_kernel(const float* __restrict__ hbuf, int H, int I,
                                                         ExpertWeights w, RouteBufs rb, float* __restrict__ partial,
                                                         int* status, int layer) {
    const int a = blockIdx.y;
    if (a >= rb.active[0]) return;
    const int e = rb.active[1 + a];
    const int beg = rb.offsets[e], n = rb.counts[e];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nblk = I / kMxBlock;
    for (int rr = 0; rr < 4; ++rr) {
        const int r = blockIdx.x * 32 + warp * 4 + rr;
        const size_t row = (size_t)e * H + r;
        const uint4* dq = reinterpret_cast<const uint4*>(w.down_q + row * (I / 2));
        const uint8_t* ds = w.down_s + row * nblk;
        for (int i0 = 0; i0 < n; i0 += 8) {
            const int ni = min(8, n - i0);
            float ad[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ad[i] = 0.0f;
            for (int blk = lane; blk < nblk; blk += 32) {
                const uint4 q = __ldg(dq + blk);
                const uint32_t sb = ds[blk];
                if (sb == 0xFFu) raise_status(status, MOE_ERR_BAD_SCALE, layer * 65536 + e);
                const float sc = e8m0_to_f32(sb);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < ni)
                        ad[i] = fmaf(dot32_e2m1(q, hbuf + (size_t)(beg + i0 + i) * I + blk * kMxBlock), sc, ad[i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float d = warp_sum(ad[i]);
                if (lane == 0 && i < ni) partial[(size_t)rb.perm[beg + i0 + i] * H + r] = d;
            }
        }
    }
}

}  // namespace moe
