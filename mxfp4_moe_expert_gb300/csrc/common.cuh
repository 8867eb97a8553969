// Device-side helpers shared by the kernels of the MXFP4 MoE library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

constexpr int kMxBlock = 32;          // elements per E8M0 scale (OCP MX v1.0)
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

// Records the first device-side error of a forward in the workspace status
// block: word 0 = status code, word 1 = detail (layer * 65536 + expert).
__device__ __forceinline__ void raise_status(int* status, int code, int detail) {
    if (atomicCAS(status, 0, code) == 0) status[1] = detail;
}

// E2M1 code (low 4 bits of c) -> exact fp32 value.  The three magnitude bits
// (2 exponent, 1 mantissa) are placed at bits 24..22 of an fp32, right above
// the mantissa's top bit, which encodes value * 2^-126 for every code (codes
// 0 and 1 land on fp32 subnormals, exactly as E2M1's own subnormal does);
// the multiply by 2^126 is exact.  The sign bit moves from bit 3 to bit 31.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    const float v = __uint_as_float(((c & 7u) << 22) | ((c & 8u) << 28));
    return v * 0x1p126f;
}

// E8M0 byte b (0..254) -> 2^(b - 127).  b = 0 is the fp32 subnormal 2^-127.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Routing outputs of one layer, in the workspace.
struct RouteBufs {
    float* logits;    // [T, E]
    int* idx;         // [T, k]
    float* gate;      // [T, k]
    int* counts;      // [E]
    int* offsets;     // [E + 1]
    int* perm;        // [T * k]
    int* active;      // [E + 1]: active[0] = number of routed experts, then their ids ascending
};

}  // namespace moe
