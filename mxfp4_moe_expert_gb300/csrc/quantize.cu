// fp32 -> MXFP4 conversion (OCP Microscaling Formats v1.0, the format that
// "MiMo x TileRT", section "第一层：FP4 选择性量化", and "MiMo 把 1T 模型推到每秒千
// token", section "FP4：只量化 MoE expert", name for the expert weights:
// blocks of 32 FP4 E2M1 elements sharing one E8M0 power-of-two scale).
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

// One thread per 32-element block: scale byte from amax, then each element's
// magnitude code by round-to-nearest-even on the E2M1 grid
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}: a midpoint goes to the neighbour whose code is
// even, which gives the comparison chain below (strict '>' where the lower
// neighbour has the even code, '>=' where the upper one has), saturating at 6.
__global__ void quantize_mxfp4_kernel(const float* __restrict__ w, int64_t nblocks, uint8_t* __restrict__ q,
                                      uint8_t* __restrict__ s) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const float4* src = reinterpret_cast<const float4*>(w + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 f = src[i];
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    int byte = 127;
    if (!(amax <= 3.4028235e38f)) {
        byte = 254;                              // Inf (NaN inputs are not supported)
    } else if (amax > 0.0f) {
        byte = ilogbf(amax) - 2 + 127;          // floor(log2 amax) - emax(E2M1) + bias
        byte = byte < 0 ? 0 : (byte > 254 ? 254 : byte);
    }
    // 1 / X = 2^(127 - byte), in [2^-127, 2^127]: built from exponent bits.
    const int e = 127 - byte;                    // -127..127
    const float inv = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
    uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float a = fabsf(v[i]) * inv;      // exact: multiply by a power of two
        uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
        m |= (__float_as_uint(v[i]) >> 28) & 8u; // sign bit of w
        words[i >> 3] |= m << (4 * (i & 7));
    }
    reinterpret_cast<uint4*>(q)[b] = make_uint4(words[0], words[1], words[2], words[3]);
    s[b] = (uint8_t)byte;
}

}  // namespace moe

extern "C" int moe_mxfp4_quantize(const float* w_dev, int64_t rows, int64_t cols, uint8_t* q_dev, uint8_t* s_dev,
                                  void* stream) {
    if (!w_dev || !q_dev || !s_dev || rows < 0 || cols < 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w_dev) & 15) || (reinterpret_cast<uintptr_t>(q_dev) & 15))
        return MOE_ERR_INVALID_ARG;
    const int64_t nblocks = rows * (cols / 32);
    if (nblocks == 0) return MOE_OK;
    const int threads = 256;
    const int64_t grid = (nblocks + threads - 1) / threads;
    if (grid > 0x7FFFFFFF) return MOE_ERR_INVALID_ARG;
    moe::quantize_mxfp4_kernel<<<(unsigned)grid, threads, 0, (cudaStream_t)stream>>>(w_dev, nblocks, q_dev, s_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
