// Small per-token phases around the experts: input staging, RMSNorm, and the
// gate-weighted combine (with the residual add of a pre-norm stack).
#pragma once

#include "common.cuh"

namespace moe {

// act[t, :] = fp32(x[t, :]); with a residual stack also resid[t, :] = act[t, :].
__global__ void prep_input_kernel(const __nv_bfloat16* __restrict__ x, int n, float* __restrict__ act,
                                  float* __restrict__ resid) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float v = __bfloat162float(x[i]);
        act[i] = v;
        if (resid) resid[i] = v;
    }
}

// act[t, :] = resid[t, :] * w / sqrt(mean(resid[t, :]^2) + eps).  One block of
// 256 threads per token; fixed reduction order.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ resid,
                                                      const __nv_bfloat16* __restrict__ w, int H, float eps,
                                                      float* __restrict__ act) {
    __shared__ float red[8];
    const int t = blockIdx.x;
    const float* r = resid + (size_t)t * H;
    float s = 0.0f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) s = fmaf(r[i], r[i], s);
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += red[i];
    const float inv = 1.0f / sqrtf(tot / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) act[(size_t)t * H + i] = r[i] * inv * __bfloat162float(w[i]);
}

// out[t, h] = (resid ? resid[t, h] : 0) + sum_{j < k, idx in shard} gate[t, j] * partial[t*k + j, h],
// slots summed in order j = 0..k-1.  Writes fp32 (or bf16) y when y != NULL,
// else updates resid in place.  Grid (T, ceil(H / 1024)), 256 threads x 4 columns.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ partial, const RouteBufs rb, int H,
                                                      int k, int e_begin, int e_end, float* resid, void* y,
                                                      int y_bf16) {
    const int t = blockIdx.x;
    const int h0 = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (h0 >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int e = rb.idx[t * k + j];
        if (e < e_begin || e >= e_end) continue;
        const float g = rb.gate[t * k + j];
        const float4 p = *reinterpret_cast<const float4*>(partial + (size_t)(t * k + j) * H + h0);
        acc.x = fmaf(g, p.x, acc.x);
        acc.y = fmaf(g, p.y, acc.y);
        acc.z = fmaf(g, p.z, acc.z);
        acc.w = fmaf(g, p.w, acc.w);
    }
    const size_t o = (size_t)t * H + h0;
    if (resid) {
        const float4 r = *reinterpret_cast<const float4*>(resid + o);
        acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
        if (!y) { *reinterpret_cast<float4*>(resid + o) = acc; return; }
    }
    if (y_bf16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&a);
        v.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(y) + o) = v;
    } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + o) = acc;
    }
}

}  // namespace moe
