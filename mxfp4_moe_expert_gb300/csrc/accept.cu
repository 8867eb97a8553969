// Acceptance of a speculative verify block: how many drafted tokens the target's
// greedy predictions confirm ("MiMo 把 1T 模型推到每秒千 token", DFlash section: one
// target forward scores all drafted positions of a block, the longest agreeing prefix
// is kept and the rest discarded; its acceptance length is the number of tokens one
// verify forward yields).
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_mxfp4.h"

namespace moe {

// Orderable key of a logit (larger logit -> larger key; NaN ranks with -inf).
__device__ __forceinline__ uint32_t accept_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (v != v) u = 0xFF800000u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One block per (stream, position): target[s, i] = argmax_v logits[s, i, v], the lowest
// index among equal maxima.  Key and index are packed in 64 bits and reduced with
// max on (key, ~index).
__global__ void __launch_bounds__(256) target_argmax_kernel(const float* __restrict__ logits, int64_t V,
                                                            int32_t* __restrict__ target) {
    const int64_t row = blockIdx.x;
    const float* src = logits + row * V;
    unsigned long long best = 0ull;
    for (int64_t v = threadIdx.x; v < V; v += blockDim.x) {
        const unsigned long long cand =
            ((unsigned long long)accept_key(__ldg(src + v)) << 32) | (0xFFFFFFFFu - (uint32_t)v);
        best = cand > best ? cand : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        best = other > best ? other : best;
    }
    __shared__ unsigned long long red[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = red[w] > best ? red[w] : best;
        target[row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
    }
}

// One thread per stream: the accepted drafted tokens a = the longest m <= B - 1 with
// tokens[s, i] == target[s, i - 1] for i = 1..m; outputs a + 1 (tokens the verify
// yields) and the target's token after the accepted prefix, target[s, a].
__global__ void accept_prefix_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ target, int S,
                                     int B, int32_t* __restrict__ accepted, int32_t* __restrict__ next_token) {
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= S) return;
    int a = 0;
    while (a + 1 < B && tokens[(int64_t)s * B + a + 1] == target[(int64_t)s * B + a]) ++a;
    accepted[s] = a + 1;
    if (next_token) next_token[s] = target[(int64_t)s * B + a];
}

}  // namespace moe

extern "C" int moe_mxfp4_accept(const float* logits_dev, const int32_t* tokens_dev, int32_t num_streams,
                                int32_t block, int64_t vocab, int32_t* target_dev, int32_t* accepted_dev,
                                int32_t* next_token_dev, void* stream) {
    if (num_streams < 0 || block < 1 || vocab < 1 || vocab > 0x7FFFFFFF) return MOE_ERR_INVALID_ARG;
    if (num_streams == 0) return MOE_OK;
    if (!logits_dev || !tokens_dev || !target_dev || !accepted_dev) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t rows = (int64_t)num_streams * block;
    if (rows > 0x7FFFFFFF) return MOE_ERR_INVALID_ARG;
    moe::target_argmax_kernel<<<(unsigned)rows, 256, 0, st>>>(logits_dev, vocab, target_dev);
    moe::accept_prefix_kernel<<<(num_streams + 127) / 128, 128, 0, st>>>(tokens_dev, target_dev, num_streams, block,
                                                                        accepted_dev, next_token_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
