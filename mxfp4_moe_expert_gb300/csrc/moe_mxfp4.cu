// Host side of the C ABI declared in include/moe_mxfp4.h: validation, the
// workspace contract, and the launch sequence of a forward.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "expert_simple.cuh"
#include "expert_tc.cuh"
#include "layer_ops.cuh"
#include "pack.cuh"
#include "persist.cuh"
#include "route.cuh"

struct moe_mxfp4_handle {
    moe_mxfp4_config cfg;
    std::vector<moe_mxfp4_layer> layers;
    std::vector<moe::TcMaps> maps;    // per layer, when the tensor-core expert path applies
    bool tma = false;
    bool packed = false;               // some layer's experts are in the packed layout (tensor-core paths only)
    int persist_grid = 0;              // CTAs of the persistent forward (one per SM), 0 = unavailable
    int device = 0;
    int sm_count = 0;
    int e_begin = 0, e_end = 0;
    std::mutex host_mu;                // serialises moe_mxfp4_forward_host on this handle
    int* status_host = nullptr;        // pinned copy of the status words for moe_mxfp4_forward_host
    ~moe_mxfp4_handle() { if (status_host) cudaFreeHost(status_host); }
};

namespace {

constexpr size_t kAlign = 256;
constexpr int kDefaultTimeoutUs = 200000;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of the workspace sections for T tokens.
struct WsLayout {
    size_t status, xstage, ystage, act, resid, logits, idx, gate, counts, offsets, perm, active, hbuf, partial;
    size_t xb4, xsf, ss, tickets, hb4, hsf, items, sync, rpart, chunk0, xc4, xcs, tsc, total;
};

// Upper bound of the chunks of one layer: every routed expert contributes
// ceil(n_e / 8) chunks of its pairs, i.e. at most T*k/8 + min(E, T*k).
size_t max_chunks(const moe_mxfp4_config& c, int T) {
    const size_t pairs = (size_t)T * c.top_k;
    return (pairs + moe::kTmaTok - 1) / moe::kTmaTok + std::min<size_t>(c.num_experts, pairs);
}
size_t max_items(const moe_mxfp4_config& c, int T) {
    return max_chunks(c, T) * (size_t)(c.inter / moe::kTmaRows + c.hidden / moe::kTmaRows);
}

// Counters of the persistent forward: per layer the expert-phase queue, per-chunk done
// counters and per-expert-group router counters.  Sized for the handle's largest block,
// so that the section sits at the same place, with the same size, whatever the block.
size_t tickets_bytes(const moe_mxfp4_config& c) {
    return (size_t)moe::kMaxPersistLayers * (1 + max_chunks(c, c.max_tokens) + 32) * 4;
}

// The workspace's state words: status words, grid-barrier word, flags, state tag, phase
// timestamps and trace (16 KB), then the counters.  At rest between persistent forwards.
constexpr size_t kStatusBytes = 16384;
constexpr size_t kStateTagOffset = 32;
size_t state_bytes(const moe_mxfp4_config& c) { return kStatusBytes + tickets_bytes(c); }

WsLayout ws_layout(const moe_mxfp4_config& c, int T) {
    WsLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    const size_t H = (size_t)c.hidden, I = (size_t)c.inter, E = (size_t)c.num_experts, k = (size_t)c.top_k;
    L.status = take(kStatusBytes);   // status words, grid-barrier word, state tag, timestamps, trace
    // the persistent forward's counters follow directly: one contiguous state section
    L.tickets = take(tickets_bytes(c));
    L.xstage = take((size_t)T * H * 2);
    L.ystage = take((size_t)T * H * 4);
    L.act = take((size_t)T * H * 4);
    L.resid = take((size_t)T * H * 4);
    L.logits = take((size_t)T * E * 4);
    L.idx = take((size_t)T * k * 4);
    L.gate = take((size_t)T * k * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take((size_t)T * k * 4);
    L.active = take((E + 1) * 4);
    L.hbuf = take((size_t)T * k * I * 4);
    L.partial = take((size_t)T * k * H * 4);
    const size_t chunks = max_chunks(c, T);
    // larger blocks (routed through the workspace): 128 operand rows per chunk (the wide
    // expert phase) and the input operand gathered per chunk
    const bool gathered = !((size_t)T * k <= 64 && (size_t)T * E <= 8192);
    const int rows = gathered ? moe::TcWide::kRowsA : moe::TcSmall::kRowsA;
    L.xb4 = take(moe::xb4_bytes(T, (int)H));
    L.xsf = take(moe::xsf_bytes(T, (int)H));
    L.ss = take((size_t)T * (H / 256 + 1) * 4);
    L.hb4 = take(chunks * moe::hb4_chunk_bytes((int)I, rows));
    L.hsf = take(chunks * moe::hsf_chunk_bytes((int)I, rows));
    L.items = take(max_items(c, T) * sizeof(moe::ItemRec));
    L.sync = take((8 + chunks) * 4);   // n_items[2], queue, abort, ..., done[chunks]
    L.rpart = take((size_t)(H / 256 + 1) * T * E * 4);   // router partials per column slice / block (>= 256 columns)
    L.chunk0 = take((E + 1) * 4);
    L.xc4 = take(gathered ? chunks * (H / 256) * moe::tc_a_tile<moe::TcWide>() : 0);
    L.xcs = take(gathered ? chunks * (H / 256) * moe::tc_sfa_stage<moe::TcWide>() : 0);
    L.tsc = take((size_t)T * 4);   // per-token 1 / rms of a residual stack (larger blocks)
    L.total = o;
    return L;
}

// ---- the workspace's state section at rest ----
// A persistent forward leaves the state section as it found it (zero counters, the
// barrier word at rest), so it issues no clearing copy.  The host zeroes the section,
// and writes the state tag, the first time a handle's persistent forward meets a
// workspace, after any other forward wrote the section, and after an error was read.
// The table records which handle last left each workspace's section at rest.
std::mutex g_state_mu;
std::unordered_map<const void*, const moe_mxfp4_handle*> g_state_owner;

unsigned long long state_tag(const moe_mxfp4_handle* h) {
    return 0x6d6f652d73746174ull ^ ((unsigned long long)reinterpret_cast<uintptr_t>(h) * 0x9E3779B97F4A7C15ull) ^
           (unsigned long long)state_bytes(h->cfg);
}

__global__ void state_init_kernel(uint4* base, size_t n16, unsigned long long tag) {
    for (size_t i = threadIdx.x; i < n16; i += blockDim.x) base[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x == 0) reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(base) + kStateTagOffset)[0] = tag;
}

// Zeroes the state section of ws and writes h's tag, unless h's persistent forward left
// it at rest (force: always).  Caller holds no lock.
int state_to_rest(const moe_mxfp4_handle* h, char* ws, cudaStream_t st, bool force) {
    std::lock_guard<std::mutex> lock(g_state_mu);
    auto it = g_state_owner.find(ws);
    if (!force && it != g_state_owner.end() && it->second == h) return MOE_OK;
    state_init_kernel<<<1, 512, 0, st>>>(reinterpret_cast<uint4*>(ws), state_bytes(h->cfg) / 16, state_tag(h));
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    // a launch captured into a graph has not run: the section is at rest only once it does
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MOE_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return MOE_OK;
    if (g_state_owner.size() >= 4096) g_state_owner.clear();   // forgetting only costs a re-zeroing
    g_state_owner[ws] = h;
    return MOE_OK;
}

// Another forward path writes the state section of ws: its next persistent forward re-zeroes it.
void state_forget(const void* ws) {
    std::lock_guard<std::mutex> lock(g_state_mu);
    g_state_owner.erase(ws);
}

// After an error was read from ws: re-zero the state section if h's persistent forward owns it.
void state_after_error(const moe_mxfp4_handle* h, char* ws, cudaStream_t st) {
    bool owned;
    {
        std::lock_guard<std::mutex> lock(g_state_mu);
        auto it = g_state_owner.find(ws);
        owned = it != g_state_owner.end() && it->second == h;
    }
    if (owned) state_to_rest(h, ws, st, true);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int check_layer(const moe_mxfp4_config& c, const moe_mxfp4_layer& l) {
    if (!l.router_w_dev || !aligned16(l.router_w_dev) || !is_device_ptr(l.router_w_dev)) return MOE_ERR_INVALID_ARG;
    // the experts: the canonical pointers, or the packed buffer (then the canonical ones may be NULL)
    const void* experts[] = {l.gate_q_dev, l.gate_s_dev, l.up_q_dev, l.up_s_dev, l.down_q_dev, l.down_s_dev};
    for (const void* p : experts)
        if (l.packed_dev ? (p && !aligned16(p)) : (!p || !aligned16(p) || !is_device_ptr(p))) return MOE_ERR_INVALID_ARG;
    if (l.packed_dev && ((reinterpret_cast<uintptr_t>(l.packed_dev) & 255) || !is_device_ptr(l.packed_dev)))
        return MOE_ERR_INVALID_ARG;
    if (l.router_b_dev && ((reinterpret_cast<uintptr_t>(l.router_b_dev) & 3) || !is_device_ptr(l.router_b_dev)))
        return MOE_ERR_INVALID_ARG;
    if (c.flags & MOE_FLAG_NORM) {
        if (!l.norm_w_dev || !aligned16(l.norm_w_dev) || !is_device_ptr(l.norm_w_dev)) return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2D uint8 tensor [rows, row_bytes] with boxes of box_x bytes x box_y rows.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_x, bool swizzle,
               uint32_t box_y = moe::kTmaRows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_maps(const moe_mxfp4_config& c, const moe_mxfp4_layer& l, moe::TcMaps* m) {
    const uint64_t H = c.hidden, I = c.inter, E = c.num_experts;
    // codes: [128 B x 128 rows] boxes (one 256-element stage), 128-byte swizzle;
    // scales: boxes of scale_box_width(K) bytes (several stages) x 128 rows
    const uint32_t wh = moe::scale_box_width((int)H), wi = moe::scale_box_width((int)I);
    m->packed = l.packed_dev ? 1 : 0;
    m->down_row0 = 0;
    if (l.packed_dev) {   // tile-major sections (pack.cuh): one box = one contiguous stage or scale group
        const moe::PackLayout P = moe::pack_layout((int)H, (int)I, (int)E);
        const uint8_t* b = l.packed_dev;
        m->down_row0 = (int)(P.down_codes / 128);
        const bool ok = encode_2d(&m->gate_q, b + P.codes, 128, (P.scales_gu - P.codes) / 128, 128, true, 256) &&
                        encode_2d(&m->gate_s, b + P.scales_gu, 128, 2 * E * I * (H / 32) / 128, 128, false, 2 * wh) &&
                        encode_2d(&m->down_s, b + P.scales_d, 128, E * H * (I / 32) / 128, 128, false, 2 * wi);
        m->up_q = m->down_q = m->gate_q;   // unused with the packed layout; valid maps all the same
        m->up_s = m->gate_s;
        return ok;
    }
    return encode_2d(&m->gate_q, l.gate_q_dev, H / 2, E * I, 128, true) &&
           encode_2d(&m->up_q, l.up_q_dev, H / 2, E * I, 128, true) &&
           encode_2d(&m->down_q, l.down_q_dev, I / 2, E * H, 128, true) &&
           encode_2d(&m->gate_s, l.gate_s_dev, H / 32, E * I, wh, false) &&
           encode_2d(&m->up_s, l.up_s_dev, H / 32, E * I, wh, false) &&
           encode_2d(&m->down_s, l.down_s_dev, I / 32, E * H, wi, false);
}

moe::RouteBufs route_bufs(char* ws, const WsLayout& L) {
    moe::RouteBufs rb;
    rb.logits = reinterpret_cast<float*>(ws + L.logits);
    rb.idx = reinterpret_cast<int*>(ws + L.idx);
    rb.gate = reinterpret_cast<float*>(ws + L.gate);
    rb.counts = reinterpret_cast<int*>(ws + L.counts);
    rb.offsets = reinterpret_cast<int*>(ws + L.offsets);
    rb.perm = reinterpret_cast<int*>(ws + L.perm);
    rb.active = reinterpret_cast<int*>(ws + L.active);
    return rb;
}

void copy_debug(const moe_mxfp4_debug* dbg, int l, int T, int E, int k, const moe::RouteBufs& rb, cudaStream_t st) {
    if (!dbg) return;
    auto cp = [&](void* dst, size_t per_layer, const void* src) {
        if (dst)
            cudaMemcpyAsync(static_cast<char*>(dst) + per_layer * l, src, per_layer, cudaMemcpyDeviceToDevice, st);
    };
    cp(dbg->topk_idx_dev, (size_t)T * k * 4, rb.idx);
    cp(dbg->topk_gate_dev, (size_t)T * k * 4, rb.gate);
    cp(dbg->expert_counts_dev, (size_t)E * 4, rb.counts);
    cp(dbg->expert_offsets_dev, (size_t)(E + 1) * 4, rb.offsets);
    cp(dbg->perm_dev, (size_t)T * k * 4, rb.perm);
}

// Multi-kernel forward: one launch per phase and per layer.
int forward_multi_kernel(moe_mxfp4_handle* h, const void* x, int T, void* y, char* ws, const WsLayout& L,
                         cudaStream_t st, const moe_mxfp4_debug* dbg) {
    const moe_mxfp4_config& c = h->cfg;
    const int H = c.hidden, I = c.inter, E = c.num_experts, k = c.top_k;
    const bool norm = (c.flags & MOE_FLAG_NORM) != 0;
    const int y_bf16 = (c.flags & MOE_FLAG_OUT_BF16) ? 1 : 0;
    int* status = reinterpret_cast<int*>(ws + L.status);
    float* act = reinterpret_cast<float*>(ws + L.act);
    float* resid = norm ? reinterpret_cast<float*>(ws + L.resid) : nullptr;
    float* hbuf = reinterpret_cast<float*>(ws + L.hbuf);
    float* partial = reinterpret_cast<float*>(ws + L.partial);
    const moe::RouteBufs rb = route_bufs(ws, L);
    const int max_active = std::min(E, T * k);
    const int n = T * H;

    moe::prep_input_kernel<<<std::min((n + 255) / 256, 4 * h->sm_count), 256, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(x), n, act, resid);
    const size_t sel_smem = (size_t)(33 * E + 64) * sizeof(int);
    for (int l = 0; l < c.num_layers; ++l) {
        const moe_mxfp4_layer& ly = h->layers[l];
        if (norm)
            moe::rmsnorm_kernel<<<T, 256, 0, st>>>(resid, reinterpret_cast<const __nv_bfloat16*>(ly.norm_w_dev), H,
                                                   c.rms_eps, act);
        moe::route_logits_kernel<<<(E + 7) / 8, 256, 0, st>>>(
            act, T, H, reinterpret_cast<const __nv_bfloat16*>(ly.router_w_dev), ly.router_b_dev, E, rb.logits);
        moe::route_select_kernel<<<1, 1024, sel_smem, st>>>(rb.logits, T, E, k, h->e_begin, h->e_end, rb);
        const moe::ExpertWeights w{ly.gate_q_dev, ly.gate_s_dev, ly.up_q_dev, ly.up_s_dev, ly.down_q_dev, ly.down_s_dev};
        if (dbg && dbg->expert_events) cudaEventRecord(static_cast<cudaEvent_t>(dbg->expert_events[2 * l]), st);
        moe::gateup_simple_kernel<<<dim3(I / 32, max_active), 256, 0, st>>>(act, H, I, k, w, rb, hbuf, status, l);
        moe::down_simple_kernel<<<dim3(H / 32, max_active), 256, 0, st>>>(hbuf, H, I, w, rb, partial, status, l);
        if (dbg && dbg->expert_events) cudaEventRecord(static_cast<cudaEvent_t>(dbg->expert_events[2 * l + 1]), st);
        const bool last = l == c.num_layers - 1;
        moe::combine_kernel<<<dim3(T, (H + 1023) / 1024), 256, 0, st>>>(partial, rb, H, k, h->e_begin, h->e_end,
                                                                        resid, last ? y : nullptr, y_bf16);
        copy_debug(dbg, l, T, E, k, rb, st);
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Work list / counters of a forward in the workspace.
moe::WorkList work_list(char* ws, const WsLayout& L) {
    int* sync = reinterpret_cast<int*>(ws + L.sync);
    moe::WorkList wl;
    wl.items = reinterpret_cast<moe::ItemRec*>(ws + L.items);
    wl.n_items = sync;
    wl.queue = sync + 2;
    wl.abort = sync + 3;
    wl.done = sync + 8;
    wl.chunk0 = reinterpret_cast<int*>(ws + L.chunk0);
    return wl;
}

// Expert-phase arguments shared by both tensor-core paths (per-layer fields set by the caller).
moe::TcArgs tc_args(const moe_mxfp4_handle* h, int T, char* ws, const WsLayout& L) {
    const moe_mxfp4_config& c = h->cfg;
    moe::TcArgs a;
    std::memset(&a, 0, sizeof(a));
    a.H = c.hidden;
    a.I = c.inter;
    a.T = T;
    a.xb4 = reinterpret_cast<const uint8_t*>(ws + L.xb4);
    a.xsf = reinterpret_cast<const uint8_t*>(ws + L.xsf);
    a.hb4 = reinterpret_cast<uint8_t*>(ws + L.hb4);
    a.hsf = reinterpret_cast<uint8_t*>(ws + L.hsf);
    a.partial = reinterpret_cast<float*>(ws + L.partial);
    a.status = reinterpret_cast<int*>(ws + L.status);
    a.timeout_ns = (unsigned long long)c.timeout_us * 1000ull;
    a.debug_stall = (c.flags & MOE_FLAG_DEBUG_STALL) ? 1 : 0;
    a.trace = nullptr;
    return a;
}

// Forward with the tensor-core expert kernel, one launch per phase: per layer the
// input staging (+ operand), router slices, top-k and grouping, the work list, one
// persistent expert launch, the combine.
int forward_tma(moe_mxfp4_handle* h, const void* x, int T, void* y, char* ws, const WsLayout& L, cudaStream_t st,
                const moe_mxfp4_debug* dbg) {
    const moe_mxfp4_config& c = h->cfg;
    const int H = c.hidden, I = c.inter, E = c.num_experts, k = c.top_k;
    const bool norm = (c.flags & MOE_FLAG_NORM) != 0;
    const int y_bf16 = (c.flags & MOE_FLAG_OUT_BF16) ? 1 : 0;
    float* act = reinterpret_cast<float*>(ws + L.act);
    float* resid = norm ? reinterpret_cast<float*>(ws + L.resid) : nullptr;
    const moe::RouteBufs rb = route_bufs(ws, L);
    const moe::WorkList wl = work_list(ws, L);
    moe::TcArgs ta = tc_args(h, T, ws, L);
    ta.items = wl.items;
    ta.n_items = wl.n_items;
    ta.queue = wl.queue;
    ta.done = wl.done;
    ta.abort = wl.abort;
    uint8_t* xb4 = reinterpret_cast<uint8_t*>(ws + L.xb4);
    uint8_t* xsf = reinterpret_cast<uint8_t*>(ws + L.xsf);
    const size_t sel_smem = (size_t)(33 * E + 64) * sizeof(int);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
    if (norm)   // r_0 = x
        moe::prep_layer_kernel<<<T, moe::kPrepThreads, 0, st>>>(xb, T, H, resid, nullptr, 0.0f, act, xb4, xsf);
    for (int l = 0; l < c.num_layers; ++l) {
        const moe_mxfp4_layer& ly = h->layers[l];
        moe::prep_layer_kernel<<<T, moe::kPrepThreads, 0, st>>>(
            xb, T, H, resid, norm ? reinterpret_cast<const __nv_bfloat16*>(ly.norm_w_dev) : nullptr, c.rms_eps, act,
            xb4, xsf);
        float* rpart = reinterpret_cast<float*>(ws + L.rpart);
        moe::route_partial_kernel<<<dim3((E + 31) / 32, H / moe::kRouteSlice), 256, 0, st>>>(
            act, T, H, reinterpret_cast<const __nv_bfloat16*>(ly.router_w_dev), E, rpart);
        moe::route_select_kernel<<<1, 1024, sel_smem, st>>>(rb.logits, T, E, k, h->e_begin, h->e_end, rb, rpart,
                                                             H / moe::kRouteSlice, ly.router_b_dev);
        moe::build_items_kernel<<<1, 1024, (size_t)T * k * sizeof(int), st>>>(rb, H, I, k, wl, T);
        ta.layer = l;
        ta.trace = (l == 0 && (c.flags & MOE_FLAG_TRACE)) ? reinterpret_cast<unsigned long long*>(ws + L.status + 4096)
                                                         : nullptr;
        if (dbg && dbg->expert_events) cudaEventRecord(static_cast<cudaEvent_t>(dbg->expert_events[2 * l]), st);
        moe::expert_tc_kernel<<<h->sm_count, moe::kTcThreads, moe::kTcSmemBytes, st>>>(h->maps[l], ta);
        if (dbg && dbg->expert_events) cudaEventRecord(static_cast<cudaEvent_t>(dbg->expert_events[2 * l + 1]), st);
        const bool last = l == c.num_layers - 1;
        moe::combine_kernel<<<dim3(T, (H + 1023) / 1024), 256, 0, st>>>(ta.partial, rb, H, k, h->e_begin, h->e_end,
                                                                        resid, last ? y : nullptr, y_bf16);
        copy_debug(dbg, l, T, E, k, rb, st);
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Persistent forward: one cooperative launch per (up to) 8 layers.
int forward_persistent(moe_mxfp4_handle* h, const void* x, int T, void* y, char* ws, const WsLayout& L,
                       cudaStream_t st, const moe_mxfp4_debug* dbg) {
    const moe_mxfp4_config& c = h->cfg;
    const int H = c.hidden, E = c.num_experts, k = c.top_k;
    moe::PersistParams p;
    std::memset(&p, 0, sizeof(p));
    p.T = T; p.H = H; p.I = c.inter; p.E = E; p.k = k;
    p.e_begin = h->e_begin; p.e_end = h->e_end;
    p.y_bf16 = (c.flags & MOE_FLAG_OUT_BF16) ? 1 : 0;
    p.norm = (c.flags & MOE_FLAG_NORM) ? 1 : 0;
    p.eps = c.rms_eps;
    p.x = reinterpret_cast<const __nv_bfloat16*>(x);
    p.y = y;
    p.resid = reinterpret_cast<float*>(ws + L.resid);
    p.xb4 = reinterpret_cast<uint8_t*>(ws + L.xb4);
    p.xsf = reinterpret_cast<uint8_t*>(ws + L.xsf);
    p.ss = reinterpret_cast<float*>(ws + L.ss);
    p.rpart = reinterpret_cast<float*>(ws + L.rpart);
    p.rb = route_bufs(ws, L);
    p.wl = work_list(ws, L);
    p.ta = tc_args(h, T, ws, L);
    p.ta.items = p.wl.items;
    p.ta.n_items = p.wl.n_items;
    p.wl.abort = reinterpret_cast<int*>(ws + L.status + 24);   // cleared with the status words
    const bool small_block = (size_t)T * k <= 64 && (size_t)T * E <= 8192;   // routed in shared memory
    p.chunk = moe::kTmaTok;
    p.terms = moe::kTcTerms;
    if (!small_block) {   // larger blocks: gathered input operand, dense unless disabled
        p.ta.xc4 = reinterpret_cast<uint8_t*>(ws + L.xc4);
        p.ta.xcs = reinterpret_cast<uint8_t*>(ws + L.xcs);
        // chunks of 128 operand rows: 32 pairs x 4 terms, or 16 x 8 without the dense operand
        p.chunk = moe::kWideTok;
        if (!(c.flags & MOE_FLAG_NO_DENSE)) {
            p.chunk = moe::kDenseTok;
            p.terms = 4;
            p.ta.dense = 1;
        }
    }
    p.ta.abort = p.wl.abort;
    p.tscale = reinterpret_cast<float*>(ws + L.tsc);
    if (c.flags & MOE_FLAG_TRACE) p.ta.trace = reinterpret_cast<unsigned long long*>(ws + L.status + 4096);
    const int chunks = (int)max_chunks(c, c.max_tokens);   // the counter section's layout (tickets_bytes)
    p.chunk_stride = chunks;
    p.queues = reinterpret_cast<int*>(ws + L.tickets);
    p.dones = p.queues + moe::kMaxPersistLayers;
    p.rcnt = p.dones + (size_t)moe::kMaxPersistLayers * chunks;
    // router units.  Blocks routed in shared memory: one token block, and the widest slice
    // that still gives every other SM a unit.  Larger blocks: the slice width and token
    // block with the fewest passes on the busiest CTA (ceil(units / grid) rounds of
    // ceil(rtok / tokens per pass) passes); ties go to the wider slice, then to fewer units.
    const int egroups = (E + moe::kPRouteExperts - 1) / moe::kPRouteExperts;
    p.rslice = 256;
    p.rtok = T;
    for (int w = 1024; w >= 512; w /= 2) {
        if (H % w == 0 && egroups * (H / w) >= h->persist_grid / 2) {
            p.rslice = w;
            break;
        }
    }
    if (!small_block) {
        long best = -1, best_units = 0;
        for (int w = 1024; w >= 256; w /= 2) {
            if (H % w) continue;
            const int tp = moe::kPRouteTok * 4 * (w >= 1024 ? 1 : 2);   // tokens per pass (router_groups)
            for (int rt = tp; rt < T + tp; rt += tp) {
                const long units = (long)egroups * (H / w) * ((T + rt - 1) / rt);
                const long cost = ((units + h->persist_grid - 1) / h->persist_grid) * ((rt + tp - 1) / tp);
                if (best < 0 || cost < best || (cost == best && w == p.rslice && units < best_units)) {
                    best = cost;
                    best_units = units;
                    p.rslice = w;
                    p.rtok = rt;
                }
            }
        }
    }
    // a single layer on a block of at most 8 tokens: whole-row router units of F experts when
    // x and F weight rows fit in the slot area (no cross-CTA sum of column slices)
    p.rfull = 0;
    if (!p.norm && small_block && T <= moe::kPRouteTok) {
        const int F = (E + h->persist_grid - 1) / h->persist_grid;
        const size_t row = (size_t)H * 2 + 16;
        const size_t need = ((size_t)T * row + 1023) / 1024 * 1024 + (size_t)F * row;
        if (need <= (size_t)moe::kTcStages * moe::kTcSlotBytes) p.rfull = F;
    }
    p.bar = reinterpret_cast<unsigned*>(ws + L.status + 16);
    p.route_flag = reinterpret_cast<int*>(ws + L.status + 20);
    p.tstamp = reinterpret_cast<unsigned long long*>(ws + L.status + 64);
    p.state_tag = reinterpret_cast<const unsigned long long*>(ws + L.status + kStateTagOffset);
    p.tag = state_tag(h);
    if (dbg) {
        p.dbg.idx = dbg->topk_idx_dev;
        p.dbg.gate = dbg->topk_gate_dev;
        p.dbg.counts = dbg->expert_counts_dev;
        p.dbg.offsets = dbg->expert_offsets_dev;
        p.dbg.perm = dbg->perm_dev;
    }
    // the state section is at rest (every launch returns it there), so nothing is cleared here
    if (const int r = state_to_rest(h, ws, st, false)) return r;
    for (int l0 = 0; l0 < c.num_layers; l0 += moe::kMaxPersistLayers) {
        const int nl = std::min(moe::kMaxPersistLayers, c.num_layers - l0);
        p.L = nl;
        p.layer_base = l0;
        p.init_from_x = l0 == 0 ? 1 : 0;
        p.write_y = (l0 + nl == c.num_layers) ? 1 : 0;
        for (int l = 0; l < nl; ++l) {
            const moe_mxfp4_layer& ly = h->layers[l0 + l];
            p.layer[l].maps = h->maps[l0 + l];
            p.layer[l].router_w = reinterpret_cast<const __nv_bfloat16*>(ly.router_w_dev);
            p.layer[l].router_b = ly.router_b_dev;
            p.layer[l].norm_w = reinterpret_cast<const __nv_bfloat16*>(ly.norm_w_dev);
        }
        void* kargs[] = {&p};
        // blocks routed through the workspace run the wide instantiation
        const void* kern =
            p.norm ? (!small_block ? reinterpret_cast<const void*>(moe::persist_kernel<true, true>)
                                   : reinterpret_cast<const void*>(moe::persist_kernel<false, true>))
                   : (!small_block ? reinterpret_cast<const void*>(moe::persist_kernel<true, false>)
                                   : reinterpret_cast<const void*>(moe::persist_kernel<false, false>));
        if (cudaLaunchCooperativeKernel(kern, dim3(h->persist_grid),
                                        dim3(moe::kTcThreads), kargs, moe::kTcSmemBytes, st) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* moe_mxfp4_status_string(int s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported device or shape";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_BAD_SCALE: return "E8M0 scale byte 0xFF (NaN) in a routed expert";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

int moe_mxfp4_create(const moe_mxfp4_config* cfg, const moe_mxfp4_layer* layers, moe_mxfp4_handle** out) {
    if (!cfg || !layers || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const moe_mxfp4_config& c = *cfg;
    if (c.num_layers < 1 || (c.num_layers > 1 && !(c.flags & MOE_FLAG_NORM))) return MOE_ERR_INVALID_ARG;
    if (c.hidden <= 0 || c.hidden % 128 || c.hidden > 16384) return MOE_ERR_INVALID_ARG;
    if (c.inter <= 0 || c.inter % 128 || c.inter > 16384) return MOE_ERR_INVALID_ARG;
    if (c.num_experts < 1 || c.num_experts > moe::kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (c.top_k < 1 || c.top_k > c.num_experts || c.top_k > moe::kMaxTopK) return MOE_ERR_INVALID_ARG;
    if (c.max_tokens < 1 || c.max_tokens > 4096) return MOE_ERR_INVALID_ARG;
    if ((c.flags & MOE_FLAG_NORM) && !(c.rms_eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (c.timeout_us < 0) return MOE_ERR_INVALID_ARG;
    int eb = c.expert_begin, ee = c.expert_end;
    if (eb == 0 && ee == 0) ee = c.num_experts;
    if (eb < 0 || ee > c.num_experts || eb >= ee) return MOE_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;
    for (int l = 0; l < c.num_layers; ++l) {
        const int r = check_layer(c, layers[l]);
        if (r != MOE_OK) return r;
    }
    const size_t sel_smem = (size_t)(33 * c.num_experts + 64) * sizeof(int);
    if (cudaFuncSetAttribute(moe::route_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem) !=
        cudaSuccess)
        return MOE_ERR_CUDA;

    bool any_packed = false;
    for (int l = 0; l < c.num_layers; ++l) any_packed |= layers[l].packed_dev != nullptr;
    // the tensor-core expert path takes K = H and K = I in 256-element stages whose
    // scale boxes are multiples of 16 bytes (K a multiple of 512); packed experts need it
    if (any_packed && ((c.hidden % 512) || (c.inter % 512))) return MOE_ERR_UNSUPPORTED;
    moe_mxfp4_handle* h = new (std::nothrow) moe_mxfp4_handle();
    if (!h) return MOE_ERR_INVALID_ARG;
    h->tma = (c.hidden % 512 == 0) && (c.inter % 512 == 0);
    if (h->tma) {
        h->maps.resize(c.num_layers);
        for (int l = 0; l < c.num_layers && h->tma; ++l) h->tma = make_maps(c, layers[l], &h->maps[l]);
        if (h->tma && cudaFuncSetAttribute(moe::expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           moe::kTcSmemBytes) != cudaSuccess) {
            delete h;
            return MOE_ERR_CUDA;
        }
        if (h->tma && cudaFuncSetAttribute(moe::build_items_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(std::min<size_t>((size_t)c.max_tokens * c.top_k, 512u * moe::kTmaTok) *
                                                 sizeof(int))) != cudaSuccess)
            h->tma = false;
        const void* persist_kernels[] = {reinterpret_cast<const void*>(moe::persist_kernel<false, false>),
                                         reinterpret_cast<const void*>(moe::persist_kernel<true, false>),
                                         reinterpret_cast<const void*>(moe::persist_kernel<false, true>),
                                         reinterpret_cast<const void*>(moe::persist_kernel<true, true>)};
        bool persist_ok = h->tma;
        for (const void* k : persist_kernels)
            persist_ok = persist_ok && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                            moe::kTcSmemBytes) == cudaSuccess;
        if (persist_ok) {
            int coop = 0;
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
            // one CTA per SM for every instantiation (they share the launch configuration)
            bool fits = coop != 0;
            for (const void* k : persist_kernels) {
                int per_sm = 0;
                fits = fits && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, moe::kTcThreads,
                                                                             moe::kTcSmemBytes) == cudaSuccess &&
                       per_sm >= 1;
            }
            if (fits) h->persist_grid = prop.multiProcessorCount;
        }
        cudaGetLastError();
    }
    if (any_packed && !h->tma) {   // packed experts are read by the tensor-core paths only
        delete h;
        return MOE_ERR_CUDA;
    }
    h->packed = any_packed;
    h->cfg = c;
    if (h->cfg.timeout_us == 0) h->cfg.timeout_us = kDefaultTimeoutUs;
    h->layers.assign(layers, layers + c.num_layers);
    h->device = dev;
    h->sm_count = prop.multiProcessorCount;
    h->e_begin = eb;
    h->e_end = ee;
    *out = h;
    return MOE_OK;
}

int moe_mxfp4_workspace_bytes(const moe_mxfp4_handle* h, int32_t num_tokens, size_t* bytes) {
    if (!h || !bytes || num_tokens < 0 || num_tokens > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(h->cfg, num_tokens).total;
    return MOE_OK;
}

int moe_mxfp4_forward(moe_mxfp4_handle* h, const void* x_dev, int32_t num_tokens, void* y_dev, void* workspace_dev,
                      size_t workspace_bytes, void* stream, const moe_mxfp4_debug* dbg) {
    if (!h || num_tokens < 0 || num_tokens > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (!x_dev || !y_dev || !aligned16(x_dev) || !aligned16(y_dev)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(h->cfg, num_tokens);
    if (!workspace_dev || (reinterpret_cast<uintptr_t>(workspace_dev) % kAlign) || workspace_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace_dev);
    const bool tma_fits = num_tokens * h->cfg.top_k <= 512 * moe::kTmaTok;
    if (h->packed && !tma_fits) return MOE_ERR_UNSUPPORTED;   // the fallback path reads canonical experts
    // the TMA work-item code holds up to 512 token chunks of 8 per expert (and the wide
    // expert phase's records hold pair ids as 16-bit halves)
    static_assert(512 * moe::kTmaTok <= 65536, "pair ids of the persistent path fit 16 bits");
    if (h->tma && num_tokens * h->cfg.top_k <= 512 * moe::kTmaTok) {
        const bool events = dbg && dbg->expert_events;
        if (h->persist_grid > 0 && !(h->cfg.flags & MOE_FLAG_MULTI_KERNEL) && !events)
            return forward_persistent(h, x_dev, num_tokens, y_dev, ws, L, st, dbg);
    }
    // the per-phase paths clear the status words per forward (and with them the state tag)
    state_forget(ws);
    if (cudaMemsetAsync(ws + L.status, 0, 64, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (h->tma && num_tokens * h->cfg.top_k <= 512 * moe::kTmaTok)
        return forward_tma(h, x_dev, num_tokens, y_dev, ws, L, st, dbg);
    return forward_multi_kernel(h, x_dev, num_tokens, y_dev, ws, L, st, dbg);
}

int moe_mxfp4_forward_host(moe_mxfp4_handle* h, const void* x_host, int32_t num_tokens, void* y_host,
                           void* workspace_dev, size_t workspace_bytes, void* stream) {
    if (!h || num_tokens < 0 || num_tokens > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(h->cfg, num_tokens);
    if (!workspace_dev || (reinterpret_cast<uintptr_t>(workspace_dev) % kAlign) || workspace_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace_dev);
    const size_t xb = (size_t)num_tokens * h->cfg.hidden * 2;
    const size_t yb = (size_t)num_tokens * h->cfg.hidden * ((h->cfg.flags & MOE_FLAG_OUT_BF16) ? 2 : 4);
    if (cudaMemcpyAsync(ws + L.xstage, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
    const int r = moe_mxfp4_forward(h, ws + L.xstage, num_tokens, ws + L.ystage, workspace_dev, workspace_bytes,
                                    stream, nullptr);
    if (r != MOE_OK) return r;
    if (cudaMemcpyAsync(y_host, ws + L.ystage, yb, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    // the status words ride on the stream behind y, so one synchronisation covers both
    std::lock_guard<std::mutex> lock(h->host_mu);
    if (!h->status_host && cudaHostAlloc(reinterpret_cast<void**>(&h->status_host), 64, cudaHostAllocPortable) !=
                               cudaSuccess) {
        h->status_host = nullptr;
        return MOE_ERR_CUDA;
    }
    if (cudaMemcpyAsync(h->status_host, workspace_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    const int s0 = h->status_host[0];
    if (s0 != MOE_OK) state_after_error(h, ws, st);
    return s0;
}

int moe_mxfp4_check(moe_mxfp4_handle* h, const void* workspace_dev, void* stream) {
    if (!h || !workspace_dev) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int s[2] = {0, 0};
    if (cudaMemcpy(s, workspace_dev, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (s[0] != MOE_OK) state_after_error(h, static_cast<char*>(const_cast<void*>(workspace_dev)), st);
    return s[0];
}

void moe_mxfp4_destroy(moe_mxfp4_handle* h) {
    if (!h) return;
    {
        std::lock_guard<std::mutex> lock(g_state_mu);
        for (auto it = g_state_owner.begin(); it != g_state_owner.end();)
            it = it->second == h ? g_state_owner.erase(it) : std::next(it);
    }
    delete h;
}

}  // extern "C"

// ---- allocation-free forward ---------------------------------------------------
// For callers that may not allocate device memory when they run the layer: the
// workspace lives in this file-scope array, one per GPU that loads the library.
// Host code must not use the array's name as a pointer (on the host it only
// stands for the symbol); its device address is looked up once per device.

namespace {
static __device__ __align__(256) unsigned char g_static_workspace[MOE_MXFP4_STATIC_WORKSPACE_BYTES];
constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxStaticDevices] = {};
}  // namespace

extern "C" int moe_mxfp4_forward_static(moe_mxfp4_handle* h, const void* x_dev, int32_t num_tokens, void* y_dev,
                                        void* stream) {
    if (!h || num_tokens < 0 || num_tokens > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (num_tokens == 0) return MOE_OK;
    if (ws_layout(h->cfg, num_tokens).total > MOE_MXFP4_STATIC_WORKSPACE_BYTES) return MOE_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != h->device) return MOE_ERR_INVALID_ARG;
    if (dev < 0 || dev >= kMaxStaticDevices) return MOE_ERR_UNSUPPORTED;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return MOE_ERR_CUDA;
            g_static_ptr[dev] = p;
        }
        ws = g_static_ptr[dev];
    }
    const int r = moe_mxfp4_forward(h, x_dev, num_tokens, y_dev, ws, MOE_MXFP4_STATIC_WORKSPACE_BYTES, stream,
                                    nullptr);
    if (r != MOE_OK) return r;
    return moe_mxfp4_check(h, ws, stream);
}

// ---- the activation encoding on its own (moe_mxfp4_split_terms) -----------------------
// Each value of a 32-element block becomes a sum of E2M1 terms with per-block E8M0
// scales (split_e2m1_terms, the same device function the kernels use), so callers and
// tests can check the encoding against its error bound directly.

namespace moe {

// One warp per 32-element block (lane = element): codes[b * 32 + lane] = the element's 8
// term codes (term j in bits 4j..4j+3), scales[b * 8 + j] = term j's E8M0 byte.
__global__ void split_terms_kernel(const float* __restrict__ x, int64_t n_blocks, uint32_t* __restrict__ codes,
                                   uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < n_blocks; b += warps) {
        uint32_t sb0, sb1;
        const uint32_t c = split_e2m1_terms(x[b * 32 + lane], sb0, sb1);
        codes[b * 32 + lane] = c;
        if (lane < kTcTerms) scales[b * kTcTerms + lane] = (uint8_t)((lane < 4 ? sb0 : sb1) >> (8 * (lane & 3)));
    }
}

}  // namespace moe

extern "C" int moe_mxfp4_split_terms(const float* x_dev, int64_t n_blocks, uint32_t* codes_dev, uint8_t* scales_dev,
                                     void* stream) {
    if (n_blocks < 0 || (n_blocks > 0 && (!x_dev || !codes_dev || !scales_dev))) return MOE_ERR_INVALID_ARG;
    if (n_blocks == 0) return MOE_OK;
    const int64_t blocks = (n_blocks + 7) / 8;
    moe::split_terms_kernel<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        x_dev, n_blocks, codes_dev, scales_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
