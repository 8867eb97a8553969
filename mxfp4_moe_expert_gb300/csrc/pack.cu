// moe_mxfp4_packed_bytes / moe_mxfp4_pack: the canonical expert layout rearranged
// into the tile-major layout of pack.cuh.  A pure byte permutation: every code and
// scale byte keeps its value; only its position changes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_mxfp4.h"
#include "pack.cuh"

namespace moe {

// Codes: 256-row tiles of 128 B (one 256-K stage).  split: a tile's rows 0..127 are rows
// blk * 128 .. of src0 and rows 128..255 the same rows of src1 (gate and up); else rows
// blk * 256 .. of src0 (down).  row_bytes = K / 2.  One thread per 16-byte piece, in
// destination order.
__global__ void pack_codes_kernel(const uint8_t* __restrict__ src0, const uint8_t* __restrict__ src1,
                                  uint8_t* __restrict__ dst, int64_t nblk, int S, int64_t row_bytes, bool split) {
    const int64_t n = nblk * S * 2048;   // 2048 pieces per 32 KB tile
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i >> 11;
        const int within = (int)(i & 2047);
        const int r = within >> 3, c = within & 7;
        const int64_t blk = tile / S;
        const int st = (int)(tile % S);
        const uint8_t* src = (split && r >= 128) ? src1 : src0;
        const int64_t row = split ? blk * 128 + (r & 127) : blk * 256 + r;
        reinterpret_cast<uint4*>(dst)[i] =
            __ldg(reinterpret_cast<const uint4*>(src + row * row_bytes + (int64_t)st * 128 + c * 16));
    }
}

// Scales: per (row block, group of G stages) a tile of 256 rows x 8 G bytes, rows as for
// the codes.  row_bytes = K / 32.
__global__ void pack_scales_kernel(const uint8_t* __restrict__ src0, const uint8_t* __restrict__ src1,
                                   uint8_t* __restrict__ dst, int64_t nblk, int K, bool split) {
    const int G = pack_scale_group(K), sw = 8 * G, per_row = sw / 16;
    const int ng = K / 256 / G;
    const int64_t row_bytes = K / 32;
    const int64_t per_tile = 256 * per_row;
    const int64_t n = nblk * ng * per_tile;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / per_tile;
        const int within = (int)(i % per_tile);
        const int r = within / per_row, c = within % per_row;
        const int64_t blk = tile / ng;
        const int g = (int)(tile % ng);
        const uint8_t* src = (split && r >= 128) ? src1 : src0;
        const int64_t row = split ? blk * 128 + (r & 127) : blk * 256 + r;
        reinterpret_cast<uint4*>(dst)[i] =
            __ldg(reinterpret_cast<const uint4*>(src + row * row_bytes + (int64_t)g * sw + c * 16));
    }
}

}  // namespace moe

namespace {
bool shape_ok(int H, int I, int E) { return H > 0 && I > 0 && E > 0 && H <= 16384 && I <= 16384 && E <= 1024; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

extern "C" int moe_mxfp4_packed_bytes(int32_t hidden, int32_t inter, int32_t num_experts, size_t* bytes) {
    if (!bytes || !shape_ok(hidden, inter, num_experts)) return MOE_ERR_INVALID_ARG;
    if (hidden % 512 || inter % 512) return MOE_ERR_UNSUPPORTED;
    *bytes = moe::pack_layout(hidden, inter, num_experts).total;
    return MOE_OK;
}

extern "C" int moe_mxfp4_pack(int32_t hidden, int32_t inter, int32_t num_experts, const moe_mxfp4_layer* layer,
                              void* packed_dev, size_t packed_bytes, void* stream) {
    if (!layer || !packed_dev || !shape_ok(hidden, inter, num_experts)) return MOE_ERR_INVALID_ARG;
    if (hidden % 512 || inter % 512) return MOE_ERR_UNSUPPORTED;
    const moe::PackLayout L = moe::pack_layout(hidden, inter, num_experts);
    if (packed_bytes < L.total || !aligned(packed_dev, 256)) return MOE_ERR_INVALID_ARG;
    const uint8_t* src[6] = {layer->gate_q_dev, layer->up_q_dev, layer->down_q_dev,
                             layer->gate_s_dev, layer->up_s_dev, layer->down_s_dev};
    for (const uint8_t* p : src)
        if (!p || !aligned(p, 16)) return MOE_ERR_INVALID_ARG;
    uint8_t* dst = static_cast<uint8_t*>(packed_dev);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t E = num_experts, H = hidden, I = inter;
    const int grid = 4096, block = 256;
    moe::pack_codes_kernel<<<grid, block, 0, st>>>(src[0], src[1], dst + L.codes, E * I / 128, (int)(H / 256), H / 2,
                                                   true);
    moe::pack_codes_kernel<<<grid, block, 0, st>>>(src[2], src[2], dst + L.down_codes, E * H / 256, (int)(I / 256),
                                                   I / 2, false);
    moe::pack_scales_kernel<<<grid, block, 0, st>>>(src[3], src[4], dst + L.scales_gu, E * I / 128, (int)H, true);
    moe::pack_scales_kernel<<<grid, block, 0, st>>>(src[5], src[5], dst + L.scales_d, E * H / 256, (int)I, false);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
