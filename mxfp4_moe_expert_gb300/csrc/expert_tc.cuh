// Expert FFN on the 5th-generation tensor cores, fed by TMA.
//
// Every routed expert's gate, up and down bytes are streamed from HBM once per
// verify block: decode speed is bandwidth over bytes read ("MiMo x TileRT",
// 万亿参数推理为什么特别难).  One CTA per SM pulls work items (worklist.cuh) from a
// queue and runs them through a ring of shared-memory stages, with the roles of
// the persistent engine's warp specialisation ("MiMo 把 1T 模型推到每秒千 token",
// persistent engine kernel and warp specialization section):
//   producer (one lane)   per stage (256 weight rows x 256 K): the packed E2M1 codes
//                         (gate and up rows of a gate/up item, or 256 rows of a down
//                         item) in the 128-byte swizzled layout, as one 32 KB TMA box
//                         from the packed layout (pack.cuh) or two [128 rows x 128 B]
//                         boxes from the canonical one, and the activation operand of
//                         down items and of gathered chunks (E2M1 terms per pair,
//                         below); the weights' E8M0 scales come per group of stages
//                         through their own ring;
//   activation loaders    (3 warps) the per-token activation rows and scales of gate/up
//                         stages, by cp.async (see tc_load);
//   MMA issuer (one lane) per stage 4 block-scaled MMAs (kind::mxf4, K = 64 each):
//                         A = the activation terms (M = 128 rows: rows 8p + j of pair
//                         slot p, term j, 8 pairs with rows 64.. unused; blocks routed
//                         through the workspace fill all 128: rows 4p + j of 32 pairs x
//                         4 terms, or 8p + j of 16 x 8), B = the weights (N = 256 rows),
//                         one E8M0 scale per row and 32-element block, fp32 accumulator
//                         [128 x 256] in tensor memory;
//   scale-factor warps    rearrange the stage's scales in shared memory into the
//                         16-byte rows that tcgen05.cp puts into tensor memory, and
//                         issue those copies (3 warps);
//   epilogue warps (8)    the used lanes of the accumulator (lane quarters 0 and 1 x
//                         four column chunks, or all four quarters x two): sum each
//                         pair's term rows (shuffle reduce-scatter over the pair's
//                         lanes), then gate/up items apply SwiGLU and store h split into
//                         E2M1 terms in the down projection's operand layout; down items
//                         store fp32 per-pair partial outputs (TcSmall / TcWide below).
// One block-scaled MMA costs about the same for N = 64 as for N = 256, so the
// weights take the wide operand: 8 KB of weights per MMA.  Every TMA request moves
// whole 128-byte rows (narrower rows cost as much per request).
// The weights are exact (E2M1 x E8M0 is what the format defines); each activation x
// is replaced by the sum of t E2M1 terms with per-32 E8M0 scales, term j encoding
// the residual of terms 0..j-1; each term at least quarters the block's largest
// residual, so the sum is within 4^-t of max|x| of its block (t = 8: N(0,1) blocks reach
// ~1e-7; the dense operand t = 4), and the tensor cores add exact products in fp32.
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "route.cuh"
#include "worklist.cuh"

namespace moe {

constexpr int kTcKS = 256;                 // K per stage
constexpr int kTcStages = 4;               // ring slots (TcSmall)
constexpr int kTcTerms = 8;                // E2M1 terms per activation
constexpr int kTcRowsA = kTmaTok * kTcTerms;   // activation rows used: pair slot p, term j -> row 8p + j
constexpr int kTcN = kDownRows;            // weight rows per MMA (gate 128 | up 128, or 256 down rows)
constexpr int kTcThreads = 512;            // 16 warps
constexpr int kTcEpiWarps = 8;
constexpr int kTcSfWarps = 3;
constexpr int kTcLoaders = 3;
// slot layout (bytes): weights [256 rows x 128 B] packed E2M1 (128-byte swizzle) at 0,
// activation terms [rows x 128 B] at kSlotA, then the scale rows for tcgen05.cp (6 x [32
// rows x 16 B]: SFA g0, g1, SFB (g, half) x 4) at the geometry's kAtoms
constexpr int kSlotB = 0;
constexpr int kSlotA = 32768;
constexpr int kSlotAtoms = 40960;          // TcSmall
constexpr int kTcSlotBytes = 45056;        // TcSmall
// scale ring entry: a pair of weight-scale boxes [128 rows x up to 64 B] (at +0 and
// +kScaleBox1), then the activation rows' E8M0 scales of the same stages (at +kScaleSfa):
//   per-token gate/up items: [pair p][stage in group][8 term rows][8 blocks];
//   down items and gathered chunks: [stage][activation rows][8 blocks]
constexpr int kScaleBox1 = 8192;
constexpr int kScaleSfa = 16384;
constexpr int kTcScaleEntry = 20480;       // TcSmall
constexpr int kTcScaleRing = 2;
constexpr int kTcAuxBytes = 4096;
constexpr int kTcSmemBytes = 1024 /*align slack*/ + kTcStages * kTcSlotBytes + kTcScaleRing * kTcScaleEntry + kTcAuxBytes;
static_assert(kTcSmemBytes <= 232448, "shared memory of the expert kernel");

// The two geometries of the expert phase, one per kernel instantiation.  Warp w runs on
// SM sub-partition w % 4 and reads tensor-memory lanes 32 (w % 4) .. +31 only, so the
// epilogue warps sit on the lane quarters that hold used accumulator rows.
//   TcSmall  (blocks routed in shared memory; the one-launch-per-phase kernel): 64
//            activation rows (8 pairs x 8 terms, rows 8p + j; the MMA's rows 64..127 read
//            on into the scale rows and are never read back), a ring of 4 stages of 44 KB,
//            epilogue warps 0, 1, 4, 5, 8, 9, 12, 13 (lane quarters 0 and 1, four 32-column
//            chunks), producer 2, MMA 3, scale-factor warps 6, 7, 10, loaders 11, 14, 15.
//   TcWide   (blocks routed through the workspace): all 128 rows of the MMA (32 pairs x 4
//            terms, rows 4p + j, or 16 pairs x 8 terms), a ring of 3 stages of 52 KB,
//            epilogue warps 0..7 (two per lane quarter, 32-column chunks c and c + 2),
//            producer 8, MMA 9, scale-factor warps 10, 11, 12, loaders 13, 14, 15.  Each
//            chunk's weights pass through the SM once for twice as many pairs.
struct TcSmall {
    static constexpr bool kWide = false;
    static constexpr int kRowsA = kTcRowsA, kStages = kTcStages, kSlotBytes = kTcSlotBytes, kAtoms = kSlotAtoms;
    static constexpr int kScaleEntry = kTcScaleEntry;
    static constexpr int kProducer = 2, kMma = 3;
    static constexpr int kChunksPerEpiWarp = 1;
    __device__ static __forceinline__ int sf_index(int w) { return w == 6 ? 0 : w == 7 ? 1 : w == 10 ? 2 : -1; }
    __device__ static __forceinline__ int loader_index(int w) { return w == 11 ? 0 : w == 14 ? 1 : w == 15 ? 2 : -1; }
    __device__ static __forceinline__ bool epi_warp(int w) { return (w & 3) < 2; }
};
struct TcWide {
    static constexpr bool kWide = true;
    static constexpr int kRowsA = 128, kStages = 3, kSlotBytes = 53248, kAtoms = 49152;
    static constexpr int kScaleEntry = 24576;
    static constexpr int kProducer = 8, kMma = 9;
    static constexpr int kChunksPerEpiWarp = 2;
    __device__ static __forceinline__ int sf_index(int w) { return (w >= 10 && w < 13) ? w - 10 : -1; }
    __device__ static __forceinline__ int loader_index(int w) { return (w >= 13) ? w - 13 : -1; }
    __device__ static __forceinline__ bool epi_warp(int w) { return w < 8; }
};
// the geometry of a kernel instantiation: TcWide for blocks routed through the workspace
template <bool kWide> struct TcGeom { using type = TcSmall; };
template <> struct TcGeom<true> { using type = TcWide; };
// bytes of one stage's activation operand and of its E8M0 scales (gathered / down layout)
template <class C> constexpr int tc_a_tile() { return C::kRowsA * 128; }
template <class C> constexpr int tc_sfa_stage() { return C::kRowsA * 8; }
template <class C> constexpr int tc_smem_need() {
    return 1024 + C::kStages * C::kSlotBytes + kTcScaleRing * C::kScaleEntry + kTcAuxBytes;
}
static_assert(tc_smem_need<TcSmall>() == kTcSmemBytes && tc_smem_need<TcWide>() <= kTcSmemBytes,
              "both geometries fit the launch's shared memory");
static_assert(kSlotA + 16384 <= kTcStages * kTcSlotBytes, "the MMA's unused activation rows stay inside shared memory");
static_assert(kSlotA + tc_a_tile<TcWide>() == TcWide::kAtoms && TcWide::kAtoms + 6 * 512 <= TcWide::kSlotBytes,
              "wide slot: weights, 128 activation rows, scale rows");
static_assert(kSlotA + tc_a_tile<TcSmall>() == TcSmall::kAtoms && TcSmall::kAtoms + 6 * 512 <= TcSmall::kSlotBytes,
              "small slot: weights, 64 activation rows, scale rows");
static_assert(kScaleSfa + 8 * tc_sfa_stage<TcWide>() <= TcWide::kScaleEntry &&
              kScaleSfa + 8 * tc_sfa_stage<TcSmall>() <= TcSmall::kScaleEntry, "scale ring entries");
static_assert(TcSmall::kSlotBytes % 1024 == 0 && TcWide::kSlotBytes % 1024 == 0 && TcWide::kScaleEntry % 1024 == 0,
              "swizzled operands are 1024-aligned");
// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemAcc = 0;           // [128 lanes x 256 columns] (gate | up, or two down row blocks)
constexpr uint32_t kTmemSf = 256;          // per slot 24: SFA groups at +0, +4; SFB groups at +8, +16 (8 columns each)
constexpr uint32_t kTmemSfSlot = 24;
static_assert(kTmemSf + kTmemSfSlot * kTcStages <= kTmemCols, "tensor memory");
constexpr int kItemRing = 8;
// global activation operand layouts (bytes); a "stage" is 256 consecutive K
//   xb4: [T][H/256][8 term rows][128 B] packed E2M1, 128-byte swizzle (row phase = term)
//   xsf: [T][H/256][8 term rows][8 blocks]
//   hb4: [chunk][I/256][R rows][128 B] swizzled; hsf: [chunk][I/256][R rows][8 blocks], R =
//        the geometry's activation rows (TcSmall 64: 8p + j; TcWide 128: 4p + j or 8p + j)
//   xc4 / xcs (blocks routed through the workspace): the layer input gathered per chunk in
//   the layout of hb4 / hsf ([chunk][H/256][128 rows][128 B] / [..][8 blocks]), so a
//   gate/up stage needs one copy
__host__ __device__ constexpr size_t xb4_bytes(int T, int H) { return (size_t)T * (H / 2) * kTcTerms; }
__host__ __device__ constexpr size_t xsf_bytes(int T, int H) { return (size_t)T * (H / 32) * kTcTerms; }
__host__ __device__ constexpr size_t hb4_chunk_bytes(int I, int rows = kTcRowsA) { return (size_t)(I / 2) * rows; }
__host__ __device__ constexpr size_t hsf_chunk_bytes(int I, int rows = kTcRowsA) { return (size_t)(I / 32) * rows; }
// Width (bytes = 32-element blocks) of a weight-scale box for K: the largest
// multiple of 16 that divides K / 32 and is at most 64.
__host__ __device__ constexpr int scale_box_width(int K) {
    int w = 64;
    while (w > 16 && (K / 32) % w) w -= 16;
    return w;
}

// Tensor maps of one layer's experts.  Canonical layout: codes uint8 [rows, K/2], box
// {128 B, 128 rows}, 128-byte swizzle (two boxes per stage); scales uint8 [rows, K/32],
// box {scale_box_width(K) B, 128 rows} (two boxes per scale group).  Packed layout
// (pack.cuh): gate_q maps the whole code region as rows of 128 B, box {128 B, 256 rows}
// with 128-byte swizzle (one stage, 32 contiguous KB); gate_s / down_s map the gate/up
// and the down scale regions as rows of 128 B, box {128 B, 2 scale_box_width(K) rows}
// (one scale group of 256 weight rows, contiguous); up_q, down_q and up_s are unused.
// Both layouts put the same bytes in the same places in shared memory, except that a
// packed scale group holds its second 128 rows right after the first (at +128 sw bytes
// instead of +kScaleBox1).
struct TcMaps {
    CUtensorMap gate_q, up_q, down_q;
    CUtensorMap gate_s, up_s, down_s;
    int packed;
    int down_row0;   // packed: first 128-byte row of the down tiles in the code region
};

struct TcArgs {
    int H, I, T, layer;
    const uint8_t* xb4;
    const uint8_t* xsf;
    const uint8_t* xc4;       // per-chunk gathered input operand, or NULL (per-token copies)
    const uint8_t* xcs;
    uint8_t* hb4;
    uint8_t* hsf;
    float* partial;           // [pairs (t*k + j), H]
    const ItemRec* items;     // work list (NULL with a routing table)
    const int* n_items;
    int* queue;               // zero at the start of the phase
    int* done;                // [chunks] zero at the start of the phase
    int* abort;
    int* status;
    unsigned long long timeout_ns;
    int debug_stall;          // testing aid: chunk 0 never signals its gate/up items
    const RouteTable* rt;     // shared-memory routing table, or NULL
    unsigned long long* trace;   // [6][256] per-stage timestamps of CTA 0 (profiling), or NULL
    int dense;                // gathered chunks hold 32 pairs x 4 E2M1 terms (rows 4p + j) instead of 16 x 8
};

// Profiling aid: event `ev` of ring stage / item i of CTA 0.
__device__ __forceinline__ void tc_trace(const TcArgs& a, int ev, uint32_t i) {
    if (a.trace && blockIdx.x == 0 && i < 256u) a.trace[ev * 256 + i] = globaltimer_ns();
}

struct TcSlotMeta {
    int kind;       // kItemGateUp, kItemDown, or -1 (end of the phase)
    int stage;      // stage within the item
    int nstages;
    int sc;         // scale-box pair counter value of this stage's pair
    int sc_off;     // byte offset of the stage's 8 scale bytes within a box row
    int sc_w;       // box row width (bytes)
    int sc_last;    // last stage reading that pair
    int pad;
    int s1off;      // byte offset of the second 128 weight rows' scales in the entry
    int ri;         // item ring entry of the stage's item (its tokens)
};

struct TcItemInfo {
    int kind, e, chunk, rb, ntok, pad0, pad1, pad2;
    int ids[kMaxChunk];   // gate/up: tokens; down: pair ids
};

struct TcSmem {
    uint8_t* slots;
    uint8_t* scales;    // [kTcScaleRing][entry]
    uint64_t *full, *empty, *accf, *acce, *ringf, *ringe, *sfull, *sempty, *epib, *drain;
    uint64_t *claim, *sfc, *drain2;   // slot claimed by the producer; scale factors in tensor memory; SF drain
    uint32_t* tmem_slot;
    TcSlotMeta* meta;
    TcItemInfo* ring;
    RouteTable* rt;
    float* red;   // 64 floats of scratch for the persistent kernel's block reductions
};

// Shared memory of geometry C: the ring's slots, the scale ring (contiguous after them:
// outside the expert phase the two are one scratch span), then barriers and records.
template <class C>
__device__ __forceinline__ TcSmem tc_smem(uint8_t* smem_raw) {
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    TcSmem s;
    s.slots = smem;
    s.scales = smem + C::kStages * C::kSlotBytes;
    uint8_t* aux = s.scales + kTcScaleRing * C::kScaleEntry;
    uint64_t* b = reinterpret_cast<uint64_t*>(aux);
    s.full = b; b += C::kStages;
    s.empty = b; b += C::kStages;
    s.accf = b; b += 1;
    s.acce = b; b += 1;
    s.ringf = b; b += kItemRing;
    s.ringe = b; b += kItemRing;
    s.sfull = b; b += kTcScaleRing;
    s.sempty = b; b += kTcScaleRing;
    s.epib = b; b += 1;
    s.drain = b; b += 1;
    s.claim = b; b += C::kStages;
    s.sfc = b; b += C::kStages;
    s.drain2 = b; b += 1;
    s.tmem_slot = reinterpret_cast<uint32_t*>(aux + 384);
    s.meta = reinterpret_cast<TcSlotMeta*>(aux + 400);
    s.ring = reinterpret_cast<TcItemInfo*>(aux + 640);
    s.rt = reinterpret_cast<RouteTable*>(aux + 640 + kItemRing * sizeof(TcItemInfo));
    s.red = reinterpret_cast<float*>(aux + 640 + kItemRing * sizeof(TcItemInfo) + sizeof(RouteTable));
    return s;
}
static_assert(8 * (4 * kTcStages + 2 + 2 * kItemRing + 2 * kTcScaleRing + 3) <= 384, "barriers");
static_assert(400 + kTcStages * sizeof(TcSlotMeta) <= 640, "slot metadata");
static_assert(640 + kItemRing * sizeof(TcItemInfo) + sizeof(RouteTable) + 64 * sizeof(float) <= kTcAuxBytes, "aux");

// One thread initialises the barriers; then the block synchronises.
template <class C>
__device__ __forceinline__ void tc_smem_init(const TcSmem& s) {
    for (int i = 0; i < C::kStages; ++i) {
        mbar_init(&s.full[i], 2);   // the producer (expect_tx) and the stage's activation loader
        mbar_init(&s.empty[i], 1);
    }
    mbar_init(s.accf, 1);
    mbar_init(s.acce, kTcEpiWarps);
    for (int i = 0; i < kItemRing; ++i) {
        mbar_init(&s.ringf[i], 1);
        mbar_init(&s.ringe[i], kTcEpiWarps);
    }
    for (int i = 0; i < kTcScaleRing; ++i) {
        mbar_init(&s.sfull[i], 2);   // the producer (expect_tx) and the group's activation loader
        mbar_init(&s.sempty[i], kTcSfWarps);
    }
    mbar_init(s.epib, kTcEpiWarps);
    mbar_init(s.drain, 1);
    for (int i = 0; i < C::kStages; ++i) {
        mbar_init(&s.claim[i], 1);
        mbar_init(&s.sfc[i], kTcSfWarps);
    }
    mbar_init(s.drain2, kTcSfWarps);
    fence_barrier_init();
}

// Waits on an mbarrier phase until it completes or the deadline passes (drains;
// ignores the abort flag).
__device__ __forceinline__ bool drain_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() > deadline) return false;
    return true;
}

// Waits on an mbarrier phase, bounded by a deadline; false on timeout or abort.
// The thread sleeps in try_wait between checks (it wakes when the phase completes).
#ifndef MOE_SLEEP_HINT_NS
#define MOE_SLEEP_HINT_NS 20000
#endif
constexpr uint32_t kSleepHintNs = MOE_SLEEP_HINT_NS;
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline,
                                           const int* abort) {
    while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
        if (globaltimer_ns() > deadline) return false;
        if (*reinterpret_cast<const volatile int*>(abort)) return false;
    }
    return true;
}

// The same wait for a whole warp: the warp leaves together (completion seen by all
// lanes, or timeout / abort seen by any).
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, unsigned long long deadline,
                                                const int* abort) {
    for (;;) {
        const bool done = mbar_try_wait_sleep(bar, parity, kSleepHintNs);
        if (__all_sync(0xFFFFFFFFu, done)) return true;
        const bool stop = globaltimer_ns() > deadline || *reinterpret_cast<const volatile int*>(abort) != 0;
        if (__any_sync(0xFFFFFFFFu, stop)) return false;
    }
}

// Splits the 32 values of one MX block (one per lane) into kTcTerms E2M1 terms:
// term j encodes the residual r left by terms 0..j-1 as codes c with r ~ c * X,
// X the power of two with max|r| / X in (3, 6] (round to nearest even on the E2M1
// grid; a value that rounds past 6 saturates and its excess stays in the residual
// for the next term).  Its E8M0 scale byte is log2(X) + 127.  A residual that is
// zero (or below 2^-120) gives zero codes and scale byte 0.  Returns the codes (term
// j in bits 4j..4j+3) and, in sb0 / sb1, the scale bytes of terms 0-3 / 4-7 (term j
// in byte j % 4, the same in every lane).
// kRedux: the block max by one redux.sync (faster where many independent splits are in
// flight; the shuffle tree is faster inside the expert epilogue).  Both give the same max.
template <bool kRedux = false>
__device__ __forceinline__ uint32_t split_e2m1_terms(float v, uint32_t& sb0, uint32_t& sb1) {
    uint32_t codes = 0;
    sb0 = sb1 = 0;
    float r = v;
#pragma unroll
    for (int j = 0; j < kTcTerms; ++j) {
        // max |r| over the block, NaNs ignored (as fmaxf does); the bits of non-negative
        // floats order like unsigned integers, which lets redux.sync take the max
        float m;
        if (kRedux) {
            m = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, r != r ? 0u : __float_as_uint(fabsf(r))));
        } else {
            m = fabsf(r);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        }
        const uint32_t eb = __float_as_uint(m) >> 23;   // biased exponent of max|r| (m >= 0)
        if (eb >= 8u && eb < 255u) {
            // X = 2^(e-2) with e = eb - 127 puts max|r| / X in [4, 8); halve the ratio when it exceeds 6
            uint32_t xb = eb - 2u;
            if (m > 6.0f * __uint_as_float(xb << 23)) ++xb;
            const float X = __uint_as_float(xb << 23);
            const float inv = __uint_as_float((254u - xb) << 23);   // 1 / X
            const uint32_t c = f32_to_e2m1(r * inv);
            r = fmaf(-e2m1_code_to_f32(c), X, r);   // exact: the code is r / X rounded to the E2M1 grid
            codes |= c << (4 * j);
            if (j < 4) sb0 |= xb << (8 * j); else sb1 |= xb << (8 * (j - 4));
        }
    }
    return codes;
}

// 8x8 nibble transpose inside each group of 8 lanes: lane l returns, for term
// j = l & 7, the codes of the 8 lanes (l & ~7) + 0..7 (lane i in bits 4i..4i+3).
__device__ __forceinline__ uint32_t transpose_oct(uint32_t codes, int lane) {
    const int base = lane & ~7, j = lane & 7;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t v = __shfl_sync(0xFFFFFFFFu, codes, base + i);
        w |= ((v >> (4 * j)) & 0xFu) << (4 * i);
    }
    return w;
}

// Stores the activation operand of token t, MX block kb (lane = element): codes into
// xb4, scale bytes into xsf.  Whole warp.
__device__ __forceinline__ void store_act_terms(uint8_t* xb4, uint8_t* xsf, int H, int t, int kb, int lane,
                                                uint32_t codes, uint32_t sb0, uint32_t sb1) {
    const uint32_t w = transpose_oct(codes, lane);   // term (lane & 7), elements (lane & ~7) .. +7
    const int j = lane & 7;
    const int st = kb >> 3;
    const int byte = (kb & 7) * 16 + (lane >> 3) * 4;   // within the stage's 128-byte row
    uint8_t* row = xb4 + (((size_t)t * (H / kTcKS) + st) * kTcTerms + j) * 128;
    *reinterpret_cast<uint32_t*>(row + ((((byte >> 4) ^ j) << 4) | (byte & 15))) = w;
    if (lane < kTcTerms)
        xsf[(((size_t)t * (H / kTcKS) + st) * kTcTerms + lane) * 8 + (kb & 7)] =
            (uint8_t)((lane < 4 ? sb0 : sb1) >> (8 * (lane & 3)));
}

// ---- producer (one thread) -----------------------------------------------------
// Claims items until the queue is empty, streams their stages into the ring and
// publishes an END slot.  The role state carries across phases.  Returns false on
// a timeout / abort.
struct TcRoleState {
    uint32_t it;    // ring position (producer, MMA, scale-factor warps)
    uint32_t n;     // item ring / accumulator position (producer, MMA, epilogue)
    uint32_t sc;    // scale-box pairs (producer, scale-factor warps)
    uint32_t eb;    // epilogue barrier uses
};

// Where an item's weights live: the two 128-row code boxes of a stage, their scale
// boxes, and the number of stages per scale-box pair.
struct TcItemGeom {
    const CUtensorMap *q0, *q1, *s0, *s1;
    int r0, r1, nk, spb, sw, packed;
    int y0, ys0;   // packed: the item's first code row and first scale row (rows of 128 B)
};
__device__ __forceinline__ TcItemGeom tc_item_geom(const TcMaps& maps, const ItemRec& it, int H, int I, int wgu,
                                                   int wd) {
    const bool gu = ((it.code >> 30) & 1) == kItemGateUp;
    const int rb = (it.code >> 20) & 0x3FF;
    TcItemGeom g;
    g.q0 = gu ? &maps.gate_q : &maps.down_q;
    g.q1 = gu ? &maps.up_q : &maps.down_q;
    g.s0 = gu ? &maps.gate_s : &maps.down_s;
    g.s1 = gu ? &maps.up_s : &maps.down_s;
    g.r0 = gu ? it.e * I + rb * kTmaRows : it.e * H + rb * kTcN;
    g.r1 = gu ? g.r0 : g.r0 + kTmaRows;
    g.nk = gu ? H / kTcKS : I / kTcKS;
    g.sw = gu ? wgu : wd;
    g.spb = g.sw / 8;
    g.packed = maps.packed;
    // packed: item (e, row block rb) owns nk consecutive 32 KB code tiles (256 rows of 128
    // B each) and nk / spb consecutive scale groups (2 sw rows of 128 B each)
    const int blk = gu ? it.e * (I / kTmaRows) + rb : it.e * (H / kTcN) + rb;
    g.y0 = (gu ? 0 : maps.down_row0) + blk * g.nk * 256;
    g.ys0 = blk * (g.nk / g.spb) * 2 * g.sw;
    if (g.packed) {
        g.q0 = g.q1 = &maps.gate_q;
        g.s0 = g.s1 = gu ? &maps.gate_s : &maps.down_s;
    }
    return g;
}
// Geometry C; TcWide: the gate/up items' activation operand comes per chunk (xc4 / xcs,
// one copy per stage and one per scale group) instead of per token and pair.
template <class C>
__device__ __noinline__ bool tc_produce(const TcMaps& maps, const TcArgs& a_in, const TcSmem& s_in,
                                        TcRoleState& rs_in, unsigned long long deadline) {
    // arguments and counters in registers (the caller's copies live in local memory)
    constexpr bool kGathered = C::kWide;
    constexpr uint32_t kATile = tc_a_tile<C>(), kSfa = tc_sfa_stage<C>();
    const TcArgs a = a_in;
    const TcSmem s = s_in;
    TcRoleState rs = rs_in;
    const int H = a.H, I = a.I;
    const int rbu = I / kTmaRows, rbd = H / kTcN;
    const int n_items = a.rt ? a.rt->n_chunks * (rbu + rbd) : __ldcg(a.n_items);
    const int wgu = scale_box_width(H), wd = scale_box_width(I);
    bool failed = false;
    int next_idx = atomicAdd(a.queue, 1);
    ItemRec next{};
    if (next_idx < n_items) next = a.rt ? table_item(a.rt, next_idx, rbu, rbd) : load_item(a.items + next_idx);
    const uint64_t pol = l2_evict_first_policy();
    for (;;) {
        const int idx = next_idx;
        const ItemRec cur = next;
        const bool end = idx >= n_items;
        // the following item is claimed now and its record read once this item's stages are
        // issued, so the claim's round trip overlaps them
        if (!end) next_idx = atomicAdd(a.queue, 1);
        const int kind = end ? -1 : (cur.code >> 30) & 1;
        const int rb = (cur.code >> 20) & 0x3FF;
        {   // item record for the epilogue
            const int re = rs.n % kItemRing;
            if (!wait_phase(&s.ringe[re], ((rs.n / kItemRing) & 1) ^ 1, deadline, a.abort)) { failed = true; break; }
            TcItemInfo inf;
            inf.kind = kind;
            inf.e = cur.e;
            inf.chunk = cur.chunk;
            inf.rb = rb;
            inf.ntok = end ? 0 : cur.ntok;
            inf.pad0 = inf.pad1 = inf.pad2 = 0;
#pragma unroll
            for (int q = 0; q < kMaxChunk; ++q) inf.ids[q] = cur.tok[q];
            s.ring[re] = inf;
            mbar_arrive(&s.ringf[re]);
            ++rs.n;
        }
        if (end) {
            const int slot = rs.it % C::kStages;
            if (!wait_phase(&s.empty[slot], ((rs.it / C::kStages) & 1) ^ 1, deadline, a.abort)) { failed = true; break; }
            s.meta[slot] = TcSlotMeta{-1, 0, 1, 0, 0, 0, 0, 0, 0, 0};   // its loader adds the second arrival
            mbar_arrive(&s.claim[slot]);
            mbar_arrive(&s.full[slot]);
            ++rs.it;
            break;
        }
        const bool gu = kind == kItemGateUp;
        // the two 128-row weight boxes of a stage: (gate, up) rows rb*128.. or down rows rb*256.., +128
        const TcItemGeom g = tc_item_geom(maps, cur, H, I, wgu, wd);
        const int nk = g.nk;                           // stages of the item
        const CUtensorMap* mq0 = g.q0;
        const CUtensorMap* mq1 = g.q1;
        const CUtensorMap* ms0 = g.s0;
        const CUtensorMap* ms1 = g.s1;
        const int r0 = g.r0, r1 = g.r1;
        const int sw = g.sw;                           // scale box width (bytes)
        const int spb = g.spb;                         // stages per scale-box pair
        bool h_ready = gu;
        for (int st = 0; st < nk; ++st) {
            if (!h_ready) {
                // every gate/up item of this chunk must have stored its h block (operand and
                // scales, both read by copies below)
                uint32_t spins = 0;
                while (ld_acquire_gpu(a.done + cur.chunk) < rbu) {
                    if ((++spins & 63u) == 0 &&
                        (globaltimer_ns() > deadline || *reinterpret_cast<const volatile int*>(a.abort))) {
                        failed = true;
                        break;
                    }
                }
                if (failed) break;   // nothing issued for this item yet
                fence_proxy_async_global();
                h_ready = true;
            }
            if (st % spb == 0) {   // the next pair of weight-scale boxes: blocks 8*st ..
                const int se = rs.sc % kTcScaleRing;
                if (!wait_phase(&s.sempty[se], ((rs.sc / kTcScaleRing) & 1) ^ 1, deadline, a.abort)) {
                    failed = true;
                    break;
                }
                uint8_t* sdst = s.scales + se * C::kScaleEntry;
                // the activation scales of per-token gate/up stages come from the loaders
                const uint32_t sfa_bytes = (gu && !kGathered) ? 0u : (uint32_t)spb * kSfa;
                mbar_arrive_expect_tx(&s.sfull[se], 2u * (uint32_t)sw * kTmaRows + sfa_bytes);
                if (g.packed) {   // one contiguous box: both 128-row halves of the group
                    const int ys = g.ys0 + (st / spb) * 2 * sw;
                    if (cur.pad[0] > 1) tma_load_2d(sdst, ms0, 0, ys, &s.sfull[se]);
                    else tma_load_2d_stream(sdst, ms0, 0, ys, &s.sfull[se], pol);
                } else if (cur.pad[0] > 1) {
                    tma_load_2d(sdst, ms0, st * 8, r0, &s.sfull[se]);
                    tma_load_2d(sdst + kScaleBox1, ms1, st * 8, r1, &s.sfull[se]);
                } else {
                    tma_load_2d_stream(sdst, ms0, st * 8, r0, &s.sfull[se], pol);
                    tma_load_2d_stream(sdst + kScaleBox1, ms1, st * 8, r1, &s.sfull[se], pol);
                }
                if (gu && kGathered) {   // the chunk's gathered scales of the group's stages
                    bulk_load(sdst + kScaleSfa, a.xcs + ((size_t)cur.chunk * (H / kTcKS) + st) * kSfa,
                              (uint32_t)spb * kSfa, &s.sfull[se]);
                } else if (!gu) {
                    bulk_load(sdst + kScaleSfa, a.hsf + ((size_t)cur.chunk * (I / kTcKS) + st) * kSfa,
                              (uint32_t)spb * kSfa, &s.sfull[se]);
                }
                ++rs.sc;
            }
            const int slot = rs.it % C::kStages;
            if (!wait_phase(&s.empty[slot], ((rs.it / C::kStages) & 1) ^ 1, deadline, a.abort)) { failed = true; break; }
            s.meta[slot] = TcSlotMeta{kind,  st, nk, (int)rs.sc - 1, (st % spb) * 8, sw, st % spb == spb - 1 ? 1 : 0,
                                      spb,   g.packed ? kTmaRows * sw : kScaleBox1, (int)((rs.n - 1) % kItemRing)};
            mbar_arrive(&s.claim[slot]);   // the scale-factor warps may prepare this slot now
            const uint32_t abytes = (gu && !kGathered) ? 0u : kATile;   // per-token rows: the loaders
            mbar_arrive_expect_tx(&s.full[slot], 2 * 16384 + abytes);
            tc_trace(a, 0, rs.it);
            ++rs.it;   // this slot now has copies in flight
            uint8_t* dst = s.slots + (size_t)slot * C::kSlotBytes;
            // rows shared by several chunks (pad[0] > 1) keep the normal L2 policy: the other
            // chunks read them again from L2
            if (g.packed) {   // one contiguous 32 KB box: the stage's 256 weight rows
                if (cur.pad[0] > 1) tma_load_2d(dst + kSlotB, mq0, 0, g.y0 + st * 256, &s.full[slot]);
                else tma_load_2d_stream(dst + kSlotB, mq0, 0, g.y0 + st * 256, &s.full[slot], pol);
            } else if (cur.pad[0] > 1) {
                tma_load_2d(dst + kSlotB, mq0, st * 128, r0, &s.full[slot]);
                tma_load_2d(dst + kSlotB + 16384, mq1, st * 128, r1, &s.full[slot]);
            } else {
                tma_load_2d_stream(dst + kSlotB, mq0, st * 128, r0, &s.full[slot], pol);
                tma_load_2d_stream(dst + kSlotB + 16384, mq1, st * 128, r1, &s.full[slot], pol);
            }
            if (gu && kGathered) {
                bulk_load(dst + kSlotA, a.xc4 + ((size_t)cur.chunk * (H / kTcKS) + st) * kATile, kATile, &s.full[slot]);
            } else if (!gu) {
                const size_t cs = (size_t)cur.chunk * (I / kTcKS) + st;
                bulk_load(dst + kSlotA, a.hb4 + cs * kATile, kATile, &s.full[slot]);
            }
        }
        if (failed) break;
        if (next_idx < n_items) next = a.rt ? table_item(a.rt, next_idx, rbu, rbd) : load_item(a.items + next_idx);
    }
    if (failed) {
        if (atomicExch(a.abort, 1) == 0) raise_status(a.status, MOE_ERR_TIMEOUT, a.layer * 65536);
        // every copy this CTA issued must land before the CTA exits
        const uint32_t issued = rs.it < (uint32_t)C::kStages ? rs.it : (uint32_t)C::kStages;
        for (uint32_t q = 0; q < issued; ++q) {
            const uint32_t last = rs.it - 1 - q;
            drain_phase(&s.full[last % C::kStages], (last / C::kStages) & 1, globaltimer_ns() + a.timeout_ns);
        }
        const uint32_t sissued = rs.sc < (uint32_t)kTcScaleRing ? rs.sc : (uint32_t)kTcScaleRing;
        for (uint32_t q = 0; q < sissued; ++q) {
            const uint32_t last = rs.sc - 1 - q;
            drain_phase(&s.sfull[last % kTcScaleRing], (last / kTcScaleRing) & 1, globaltimer_ns() + a.timeout_ns);
        }
    }
    rs_in = rs;
    return !failed;
}

// ---- MMA issuer (one thread) -----------------------------------------------------
template <class C>
__device__ __noinline__ bool tc_mma(const TcArgs& a_in, const TcSmem& s_in, uint32_t tmem, TcRoleState& rs_in,
                                    unsigned long long deadline) {
    const TcArgs a = a_in;
    const TcSmem s = s_in;
    TcRoleState rs = rs_in;
    constexpr uint32_t kIdesc = idesc_mxf4(128, kTcN);
    const uint32_t slots = smem_u32(s.slots);
    bool failed = false;
    for (;;) {
        const int slot = rs.it % C::kStages;
        // the stage's operands have landed and its scale factors are in tensor memory
        if (!wait_phase(&s.full[slot], (rs.it / C::kStages) & 1, deadline, a.abort) ||
            !wait_phase(&s.sfc[slot], (rs.it / C::kStages) & 1, deadline, a.abort)) {
            failed = true;
            break;
        }
        tc_fence_after();
        tc_trace(a, 3, rs.it);
        const TcSlotMeta m = s.meta[slot];
        if (m.kind < 0) {   // END: release the slot and wake the epilogue
            mbar_arrive(&s.empty[slot]);
            ++rs.it;
            if (!wait_phase(s.acce, (rs.n & 1) ^ 1, deadline, a.abort)) { failed = true; break; }
            mbar_arrive(s.accf);
            ++rs.n;
            break;
        }
        if (m.stage == 0) {   // the accumulator must have been read out
            if (!wait_phase(s.acce, (rs.n & 1) ^ 1, deadline, a.abort)) { failed = true; break; }
            tc_fence_after();
        }
        const uint32_t sl = slots + (uint32_t)slot * C::kSlotBytes;
        const uint32_t sf = tmem + kTmemSf + kTmemSfSlot * slot;
        const uint64_t ad = smem_desc_sw128(sl + kSlotA), bd = smem_desc_sw128(sl + kSlotB);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // K = 64 each: blocks 2kk, 2kk+1
            const uint32_t id = 2 * (kk & 1);
            tc_mma_mxf4(tmem + kTmemAcc, ad + 2 * kk, bd + 2 * kk, kIdesc | idesc_sf_ids(id, id), sf + 4 * (kk >> 1),
                        sf + 8 + 8 * (kk >> 1), (m.stage == 0 && kk == 0) ? 0u : 1u);
        }
        tc_commit(&s.empty[slot]);
        if (m.stage == m.nstages - 1) {
            tc_commit(s.accf);
            ++rs.n;
        }
        tc_trace(a, 4, rs.it);
        ++rs.it;
    }
    if (failed && atomicExch(a.abort, 1) == 0) raise_status(a.status, MOE_ERR_TIMEOUT, a.layer * 65536);
    rs_in = rs;
    return !failed;
}

// ---- scale-factor warps ------------------------------------------------------------
// The MMA reads activation row m's scales from lane m, column base + m / 32, and
// weight row n's scales from lane n % 32 of the reading row's quarter, column
// base + n / 32 (one 32-bit cell = 4 blocks; group g = blocks 4g..4g+3 of the
// stage).  tcgen05.cp 32x128b.warpx4 puts 16-byte row r of a 512-byte block into
// columns +0..3 of lane r of every quarter, so the six blocks of a stage are:
// SFA group g (block g), row r = cells of activation rows r, 32 + r, 64 + r, 96 + r
// (TcSmall: rows 64.. unused, zero); SFB group g, half h (block 2 + 2g + h), row r = cells of weight
// rows 128h + r, 128h + 32 + r, 128h + 64 + r, 128h + 96 + r.  Warp w = 0, 1 builds
// the SFB blocks of half h = w (both groups), warp 2 the SFA blocks; lane r builds
// row r, and lane 0 copies the warp's two blocks into the slot's tensor-memory
// columns and commits to sfc[slot] (three arrivals), which the MMA thread waits on.
// A slot is prepared as soon as the producer has claimed it (its previous MMAs are
// done): the scales come from the scale ring, not from the slot's own copies, so
// the work overlaps the stage's weight copies.
// TcWide: the activation scales of gate/up stages are gathered per chunk and laid out
// per stage, like the down items', instead of per pair.
template <class C>
__device__ __noinline__ bool tc_sf(const TcArgs& a_in, const TcSmem& s_in, uint32_t tmem, TcRoleState& rs_in, int w,
                                   int lane, unsigned long long deadline) {
    constexpr bool kGathered = C::kWide;
    constexpr int kQ = C::kRowsA / 32;   // lane quarters of used activation rows
    const TcArgs a = a_in;
    const TcSmem s = s_in;
    TcRoleState rs = rs_in;
    bool failed = false;
    for (;;) {
        const int slot = rs.it % C::kStages;
        const uint32_t ph = (rs.it / C::kStages) & 1;
        if (!warp_wait_phase(&s.claim[slot], ph, deadline, a.abort)) { failed = true; break; }
        const TcSlotMeta m = s.meta[slot];
        if (w == 0 && lane == 0) tc_trace(a, 1, rs.it);
        if (m.kind >= 0) {
            const int se = m.sc % kTcScaleRing;
            if (!warp_wait_phase(&s.sfull[se], (m.sc / kTcScaleRing) & 1, deadline, a.abort)) { failed = true; break; }
            const uint8_t* ent = s.scales + se * C::kScaleEntry;
            uint8_t* at = s.slots + (size_t)slot * C::kSlotBytes + C::kAtoms;
            int b0, b1;   // the warp's two blocks
            if (w < 2) {
                uint2 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[c] = *reinterpret_cast<const uint2*>(ent + w * m.s1off + (32 * c + lane) * m.sc_w + m.sc_off);
                uint32_t ff = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    ff |= (v[c].x & (v[c].x >> 1) & (v[c].x >> 2) & (v[c].x >> 3) & (v[c].x >> 4) & (v[c].x >> 5) &
                           (v[c].x >> 6) & (v[c].x >> 7) & 0x01010101u) |
                          (v[c].y & (v[c].y >> 1) & (v[c].y >> 2) & (v[c].y >> 3) & (v[c].y >> 4) & (v[c].y >> 5) &
                           (v[c].y >> 6) & (v[c].y >> 7) & 0x01010101u);
                if (ff) raise_status(a.status, MOE_ERR_BAD_SCALE, a.layer * 65536);   // scale byte 0xFF (NaN)
                b0 = 2 + w;
                b1 = 4 + w;
                *reinterpret_cast<uint4*>(at + b0 * 512 + lane * 16) = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
                *reinterpret_cast<uint4*>(at + b1 * 512 + lane * 16) = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
            } else {   // activation rows 32 c + lane (sg = stage within the scale group)
                const int sg = m.sc_off / 8;
                uint2 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int row = 32 * c + lane;
                    const int off = (!kGathered && m.kind == kItemGateUp)
                                        ? (row >> 3) * m.pad * 64 + sg * 64 + (row & 7) * 8
                                        : sg * tc_sfa_stage<C>() + row * 8;
                    v[c] = c < kQ ? *reinterpret_cast<const uint2*>(ent + kScaleSfa + off) : make_uint2(0u, 0u);
                }
                b0 = 0;
                b1 = 1;
                *reinterpret_cast<uint4*>(at + lane * 16) = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
                *reinterpret_cast<uint4*>(at + 512 + lane * 16) = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
            }
            fence_proxy_async_shared();   // read next by tcgen05.cp
            __syncwarp();
            if (lane == 0) {
                if (m.sc_last) mbar_arrive(&s.sempty[se]);
                const uint32_t sl = smem_u32(s.slots) + (uint32_t)slot * C::kSlotBytes + C::kAtoms;
                const uint32_t sf = tmem + kTmemSf + kTmemSfSlot * slot;
                tc_cp_32x128_x4(sf + 4 * b0, smem_desc_rows16(sl + 512 * b0));
                tc_cp_32x128_x4(sf + 4 * b1, smem_desc_rows16(sl + 512 * b1));
                tc_commit(&s.sfc[slot]);
            }
        } else if (lane == 0) {
            mbar_arrive(&s.sfc[slot]);   // END: keeps the barrier's phases in step
        }
        __syncwarp();
        if (w == 0 && lane == 0) tc_trace(a, 2, rs.it);
        ++rs.it;
        if (m.kind < 0) break;
    }
    if (failed && lane == 0 && atomicExch(a.abort, 1) == 0) raise_status(a.status, MOE_ERR_TIMEOUT, a.layer * 65536);
    rs_in = rs;
    return !failed;
}

// ---- activation loaders -----------------------------------------------------------
// The per-token activation operand of a gate/up stage (rows 8p + j of pair p: its
// token's 8 E2M1 term rows, 1 KB) and, at a scale group's first stage, the group's
// activation scales (per pair spb x 64 B) are read from global memory with 16-byte
// cp.async by a whole warp, not by the TMA producer: every CTA reads these few KB of
// hot L2 lines at about the same time, and as bulk copies they held the producer's
// queue behind them (about 0.3-0.6 us per 1 KB copy, measured).  The loader of a stage
// waits for its copies, makes them visible to the tensor cores' proxy and arrives on
// the stage's full barrier (and the group's scale barrier); for every other stage it
// arrives at once.  All loaders follow every ring position, so that each one sees the
// END slot.  TcWide: every operand comes by bulk copy (gathered per chunk); the loaders
// only arrive.
template <class C>
__device__ __noinline__ bool tc_load(const TcArgs& a_in, const TcSmem& s_in, TcRoleState& rs_in, int li, int lane,
                                     unsigned long long deadline) {
    const TcArgs a = a_in;
    const TcSmem s = s_in;
    TcRoleState rs = rs_in;
    const int nst = a.H / kTcKS;
    bool failed = false;
    for (;;) {
        const int slot = rs.it % C::kStages;
        if (!warp_wait_phase(&s.claim[slot], (rs.it / C::kStages) & 1, deadline, a.abort)) { failed = true; break; }
        const TcSlotMeta m = s.meta[slot];
        const bool mine = (int)(rs.it % kTcLoaders) == li;
        ++rs.it;
        if (!mine) {
            if (m.kind < 0) break;
            continue;
        }
        const bool first = m.kind >= 0 && m.sc_off == 0;   // the first stage of a scale group
        if (!C::kWide && m.kind == kItemGateUp && !a.xc4) {
            const TcItemInfo& inf = s.ring[m.ri];
            const int ntok = inf.ntok;
            const uint32_t dst = smem_u32(s.slots + (size_t)slot * C::kSlotBytes + kSlotA);
            for (int p = 0; p < ntok; ++p) {
                const uint8_t* src = a.xb4 + ((size_t)inf.ids[p] * nst + m.stage) * 1024;
                cp_async_16(dst + p * 1024 + lane * 16, src + lane * 16);
                cp_async_16(dst + p * 1024 + 512 + lane * 16, src + 512 + lane * 16);
            }
            if (first) {   // the group's activation scales: per pair spb stages x 64 B, contiguous in xsf
                const uint32_t sdst = smem_u32(s.scales + (m.sc % kTcScaleRing) * C::kScaleEntry + kScaleSfa);
                const int per = m.pad * 4;   // 16-byte pieces per pair (spb x 64 B)
                for (int i = lane; i < ntok * per; i += 32) {
                    const int p = i / per, q = i % per;
                    cp_async_16(sdst + p * m.pad * 64 + q * 16,
                                a.xsf + ((size_t)inf.ids[p] * nst + m.stage) * 64 + q * 16);
                }
            }
            cp_async_wait_all();
            fence_proxy_async_shared();   // read next by the tensor cores (and tcgen05.cp)
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&s.full[slot]);
            if (first) mbar_arrive(&s.sfull[m.sc % kTcScaleRing]);
        }
        if (m.kind < 0) break;
    }
    cp_async_wait_all();
    if (failed && lane == 0 && atomicExch(a.abort, 1) == 0) raise_status(a.status, MOE_ERR_TIMEOUT, a.layer * 65536);
    rs_in = rs;
    return !failed;
}

// Reduce-scatter of 32 values over the 8 lanes of each lane group (lane & 7): lane
// j returns the group sums of values j, j + 8, j + 16, j + 24 (halving butterfly,
// partner offsets 4, 2, 1; a fixed order, the same on every run).
__device__ __forceinline__ void group8_reduce_scatter(const float (&v)[32], float (&out)[4], int lane) {
    float a16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {   // keep values with bit 2 of the index == bit 2 of the lane
        const int k0 = (i & 3) | ((i >> 2) << 3), k1 = k0 | 4;   // pairs differing in bit 2
        const bool hi = (lane & 4) != 0;
        const float send = hi ? v[k0] : v[k1], keep = hi ? v[k1] : v[k0];
        a16[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
    }
    // a16[i] now stands for index k = (i & 3) | (bit2 of lane) << 2 | (i >> 2) << 3
    float a8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {   // pairs differing in bit 1 of k: a16 indices (i&1) | ((i>>1)<<2) and +2
        const int i0 = (i & 1) | ((i >> 1) << 2), i1 = i0 | 2;
        const bool hi = (lane & 2) != 0;
        const float send = hi ? a16[i0] : a16[i1], keep = hi ? a16[i1] : a16[i0];
        a8[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 2);
    }
    // a8[i]: k = (i & 1) | (bit1 of lane) << 1 | (bit2 of lane) << 2 | (i >> 1) << 3
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // pairs differing in bit 0 of k: a8 indices 2i and 2i+1
        const bool hi = (lane & 1) != 0;
        const float send = hi ? a8[2 * i] : a8[2 * i + 1], keep = hi ? a8[2 * i + 1] : a8[2 * i];
        out[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 1);
    }
    // out[i]: k = (lane & 7) | i << 3
}

// The same over the 4 lanes of each lane group (lane & 3): lane j returns the group sums
// of values j + 4i, i = 0..7 (partner offsets 2, 1; a fixed order).
__device__ __forceinline__ void group4_reduce_scatter(const float (&v)[32], float (&out)[8], int lane) {
    float a16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {   // pairs differing in bit 1 of the index
        const int k0 = (i & 1) | ((i >> 1) << 2), k1 = k0 | 2;
        const bool hi = (lane & 2) != 0;
        const float send = hi ? v[k0] : v[k1], keep = hi ? v[k1] : v[k0];
        a16[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 2);
    }
    // a16[i]: k = (i & 1) | (bit1 of lane) << 1 | (i >> 1) << 2
#pragma unroll
    for (int i = 0; i < 8; ++i) {   // pairs differing in bit 0: a16 indices 2i and 2i+1
        const bool hi = (lane & 1) != 0;
        const float send = hi ? a16[2 * i] : a16[2 * i + 1], keep = hi ? a16[2 * i + 1] : a16[2 * i];
        out[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 1);
    }
    // out[i]: k = (lane & 3) | i << 2
}

// ---- epilogue warps (lane quarter q = warp % 4, 32-column chunks c) --------------
// TcSmall: warps of quarters 0 and 1, c = warp / 4; TcWide: warps 0..7, c = warp / 4 and
// warp / 4 + 2.  Each warp reads, per chunk c, columns 32c.. (gate rows / first down
// block) and 128 + 32c.. (up rows / second down block) of its 32 lanes.
// kDense = false: accumulator lane 32q + l is activation row 32q + l: pair slot 4q + l / 8,
// term l % 8; after the reduce-scatter over groups of 8 lanes, lane l holds, for its pair,
// the sums of columns 32c + 8s + (l % 8) and 128 + 32c + 8s + (l % 8), s = 0..3.
// kDense = true (4 terms): pair slot 8q + l / 4, term l % 4; lane l holds the sums of
// columns 32c + 4s + (l % 4) and 128 + .., s = 0..7.
// TcWide items carry their pairs' ids as 16-bit halves (two per word of the record).
// kNorm (residual stack): the layer input's operand is r * w_norm without the per-token
// factor 1 / rms(r), which the gate/up outputs take here, from the shared-memory routing
// table: its tscale (a.rt set: the block was routed in shared memory) or tscale_g.
template <class C, bool kDense, bool kNorm>
__device__ __noinline__ bool tc_epilogue(const TcArgs& a_in, const TcSmem& s_in, uint32_t tmem, TcRoleState& rs_in,
                                         int warp, int lane, unsigned long long deadline) {
    constexpr int kT = kDense ? 4 : kTcTerms;   // terms per activation: lanes (accumulator rows) per pair
    constexpr int kV = 32 / kT;                 // columns per lane of each 32-column chunk
    constexpr int kCW = C::kChunksPerEpiWarp;   // 32-column chunks of this warp: c0, c0 + 2
    const TcArgs a = a_in;
    const TcSmem s = s_in;
    TcRoleState rs = rs_in;
    const int q = warp & 3, c0 = warp >> 2;
    const int H = a.H, I = a.I;
    const int p = (32 / kT) * q + lane / kT, j = lane % kT;   // pair slot and term of this lane's row
    const int base = lane & ~(kT - 1);                        // first lane of the pair
    bool failed = false;
    // barrier of the epilogue warps (bounded)
    auto epi_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(s.epib);
        const bool ok = warp_wait_phase(s.epib, rs.eb & 1, deadline, a.abort);
        ++rs.eb;
        return ok;
    };
    for (;;) {
        const int re = rs.n % kItemRing;
        if (!warp_wait_phase(s.accf, rs.n & 1, deadline, a.abort) ||
            !warp_wait_phase(&s.ringf[re], (rs.n / kItemRing) & 1, deadline, a.abort)) {
            failed = true;
            break;
        }
        const int kind = s.ring[re].kind, chunk = s.ring[re].chunk, rb = s.ring[re].rb, ntok = s.ring[re].ntok;
        // this lane's pair: token (gate/up) or pair id (down)
        const int my_id = C::kWide ? (s.ring[re].ids[p >> 1] >> (16 * (p & 1))) & 0xFFFF : s.ring[re].ids[p];
        tc_fence_after();
        if (warp == 0 && lane == 0) tc_trace(a, 5, rs.n);
        const bool mine = p < ntok;
        // TcWide: a warp whose lane quarter holds no pair of the chunk has nothing to read
        // or store (its accumulator rows are never read back)
        const bool used = !C::kWide || (32 / kT) * q < ntok;
        // TcSmall: G, U = the column sums (gate / up, or the two down blocks), used after the
        // accumulator is released.  TcWide: each chunk is finished as soon as it is read, so
        // that only 8 values per chunk stay live: down items store their sums at once (the
        // stores do not wait), gate/up items keep h = silu(g) * u in G.
        float G[kCW][kV], U[kCW][kV];
        if (kind >= 0 && used) {
            if constexpr (kCW == 1) {   // both column blocks in flight at once
                uint32_t r0[32], r1[32];
                const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kTmemAcc + 32 * c0;
                tc_ld_x32(ta, r0);
                tc_ld_x32(ta + 128, r1);
                tc_wait_ld();
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r0[i]);
                if constexpr (kDense) group4_reduce_scatter(v, G[0], lane); else group8_reduce_scatter(v, G[0], lane);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r1[i]);
                if constexpr (kDense) group4_reduce_scatter(v, U[0], lane); else group8_reduce_scatter(v, U[0], lane);
            } else {
                float sc = 1.0f;   // RMSNorm(r) = (r * w_norm) / rms(r): the per-token factor
                if constexpr (kNorm)
                    if (kind == kItemGateUp && mine) sc = a.rt ? a.rt->tscale[my_id] : __ldcg(s.rt->tscale_g + my_id);
#pragma unroll
                for (int h = 0; h < kCW; ++h) {
                    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kTmemAcc + 32 * (c0 + 2 * h);
                    uint32_t r[32];
                    float v[32];
                    tc_ld_x32(ta, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    if constexpr (kDense) group4_reduce_scatter(v, G[h], lane); else group8_reduce_scatter(v, G[h], lane);
                    tc_ld_x32(ta + 128, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    if constexpr (kDense) group4_reduce_scatter(v, U[h], lane); else group8_reduce_scatter(v, U[h], lane);
                    if (kind == kItemGateUp) {
#pragma unroll
                        for (int i = 0; i < kV; ++i) G[h][i] = silu(G[h][i] * sc) * (U[h][i] * sc);
                    } else if (mine) {   // down: rows rb * 256 + 32c + kT s + j and + 128
                        float* dst = a.partial + (size_t)my_id * H + (size_t)rb * kTcN + 32 * (c0 + 2 * h) + j;
#pragma unroll
                        for (int i = 0; i < kV; ++i) {
                            dst[kT * i] = G[h][i];
                            dst[128 + kT * i] = U[h][i];
                        }
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(s.acce);
            mbar_arrive(&s.ringe[re]);
        }
        ++rs.n;
        if (kind < 0) break;
        if (kind == kItemGateUp) {
            // h = silu(g) * u for rows 32c + kT s + j of the item's 128 (s < kV); the 32 rows
            // 32c.. are one MX block of the down projection's K.  Split into kT E2M1 terms
            // with block scales over the pair's kT lanes, stored as rows kT p + t of the
            // chunk's down operand at K = rb * 128 + 32c + kT s + j.
            if constexpr (kNorm && kCW == 1) {   // g and u of RMSNorm(r) = (g and u of r * w_norm) / rms(r), per token
                const float sc = mine ? (a.rt ? a.rt->tscale[my_id] : __ldcg(s.rt->tscale_g + my_id)) : 1.0f;
#pragma unroll
                for (int i = 0; i < kV; ++i) {
                    G[0][i] *= sc;
                    U[0][i] *= sc;
                }
            }
#pragma unroll
            for (int h = 0; h < kCW; ++h) {
                if (!used) break;
                const int c = c0 + 2 * h;
                float hv[kV];
#pragma unroll
                for (int i = 0; i < kV; ++i) hv[i] = kCW == 1 ? silu(G[0][i]) * U[0][i] : G[h][i];
                uint32_t codes[kV];   // per s: term t in bits 4t..4t+3
#pragma unroll
                for (int i = 0; i < kV; ++i) codes[i] = 0u;
                uint32_t sbt = 0;     // this lane's scale byte: term j
#pragma unroll
                for (int t = 0; t < kT; ++t) {
                    float mx = 0.0f;
#pragma unroll
                    for (int i = 0; i < kV; ++i) mx = fmaxf(mx, fabsf(hv[i]));
#pragma unroll
                    for (int o = 1; o < kT; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                    const uint32_t eb = __float_as_uint(mx) >> 23;
                    if (eb >= 8u && eb < 255u) {
                        uint32_t xb = eb - 2u;
                        if (mx > 6.0f * __uint_as_float(xb << 23)) ++xb;
                        const float X = __uint_as_float(xb << 23);
                        const float inv = __uint_as_float((254u - xb) << 23);
#pragma unroll
                        for (int i = 0; i < kV; ++i) {
                            const uint32_t cd = f32_to_e2m1(hv[i] * inv);
                            hv[i] = fmaf(-e2m1_code_to_f32(cd), X, hv[i]);
                            codes[i] |= cd << (4 * t);
                        }
                        if (t == j) sbt = xb;
                    }
                }
                // lane j of the pair gathers term j's codes of the pair's kT lanes: column n (0..31)
                // of the chunk is value n / kT of lane n % kT
                uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int n = 0; n < 32; ++n) {
                    const uint32_t v = __shfl_sync(0xFFFFFFFFu, codes[n / kT], base + n % kT);
                    wd[n / 8] |= ((v >> (4 * j)) & 0xFu) << (4 * (n % 8));
                }
                if (mine) {
                    uint8_t* hb = a.hb4 + (size_t)chunk * hb4_chunk_bytes(I, C::kRowsA) + (size_t)(rb >> 1) * tc_a_tile<C>();
                    const int n = kT * p + j;                    // operand row: pair slot p, term j
                    const int chunk16 = (rb & 1) * 4 + c;        // 16-byte chunk of K (rb&1)*128 + 32c .. +31
                    *reinterpret_cast<uint4*>(hb + n * 128 + ((chunk16 ^ (n & 7)) << 4)) =
                        make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    a.hsf[(size_t)chunk * hsf_chunk_bytes(I, C::kRowsA) + (size_t)(rb >> 1) * tc_sfa_stage<C>() + n * 8 +
                          4 * (rb & 1) + c] = (uint8_t)sbt;
                }
            }
            fence_proxy_async_global();   // read next by bulk copies
            if (!epi_sync()) { failed = true; break; }
            if (warp == 0 && lane == 0 && !(a.debug_stall && chunk == 0)) {
                __threadfence();
                fence_proxy_async_global();
                red_release_add_gpu(a.done + chunk, 1);
            }
        } else if (kCW == 1 && mine) {   // down: rows rb * 256 + 32c + kT s + j and + 128
            float* dst = a.partial + (size_t)my_id * H + (size_t)rb * kTcN + 32 * c0 + j;
#pragma unroll
            for (int i = 0; i < kV; ++i) {
                dst[kT * i] = G[0][i];
                dst[128 + kT * i] = U[0][i];
            }
        }
    }
    if (failed && lane == 0 && atomicExch(a.abort, 1) == 0) raise_status(a.status, MOE_ERR_TIMEOUT, a.layer * 65536);
    rs_in = rs;
    return !failed;
}

// One expert phase of geometry C, dispatched by warp role; every thread of the block
// calls it.
template <class C, bool kNorm = false>
__device__ __forceinline__ void tc_phase(const TcMaps& maps, const TcArgs& a, const TcSmem& s, uint32_t tmem,
                                         TcRoleState& rs, unsigned long long deadline) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == C::kProducer) {
        if (lane == 0) tc_produce<C>(maps, a, s, rs, deadline);
    } else if (warp == C::kMma) {
        if (lane == 0) tc_mma<C>(a, s, tmem, rs, deadline);
    } else if (C::sf_index(warp) >= 0) {
        tc_sf<C>(a, s, tmem, rs, C::sf_index(warp), lane, deadline);
    } else if (C::loader_index(warp) >= 0) {
        tc_load<C>(a, s, rs, C::loader_index(warp), lane, deadline);
    } else if (C::epi_warp(warp)) {
        if (C::kWide && a.dense) tc_epilogue<C, true, kNorm>(a, s, tmem, rs, warp, lane, deadline);
        else tc_epilogue<C, false, kNorm>(a, s, tmem, rs, warp, lane, deadline);
    }
}

// Setup shared by the standalone and persistent kernels: barriers (thread 0) and
// the tensor-memory allocation (the MMA warp).  Ends with a block-wide barrier.
template <class C>
__device__ __forceinline__ uint32_t tc_setup(const TcSmem& s) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) tc_smem_init<C>(s);
    if (warp == C::kMma) {
        tmem_alloc(s.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *s.tmem_slot;
}

// Teardown: every tcgen05 operation of the MMA thread has completed (bounded
// wait), then the MMA warp frees the tensor memory.  All threads call it.
template <class C>
__device__ __forceinline__ void tc_teardown(const TcSmem& s, uint32_t tmem, unsigned long long timeout_ns) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == C::kMma && lane == 0) {
        tc_commit(s.drain);
        drain_phase(s.drain, 0, globaltimer_ns() + timeout_ns);
    }
    if (C::sf_index(warp) >= 0 && lane == 0) {   // the scale-factor warps' tensor-memory copies
        tc_commit(s.drain2);
        drain_phase(s.drain2, 0, globaltimer_ns() + timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMma) tmem_dealloc(tmem, kTmemCols);
}

__global__ void __launch_bounds__(kTcThreads, 1) expert_tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const TcSmem s = tc_smem<TcSmall>(smem_raw);
    const uint32_t tmem = tc_setup<TcSmall>(s);
    const unsigned long long deadline = globaltimer_ns() + args.timeout_ns;
    if (threadIdx.x == TcSmall::kProducer * 32) {
        prefetch_tensormap(&maps.gate_q);
        prefetch_tensormap(&maps.up_q);
        prefetch_tensormap(&maps.down_q);
        prefetch_tensormap(&maps.gate_s);
        prefetch_tensormap(&maps.up_s);
        prefetch_tensormap(&maps.down_s);
    }
    TcRoleState rs{0u, 0u, 0u, 0u};
    tc_phase<TcSmall>(maps, args, s, tmem, rs, deadline);
    tc_teardown<TcSmall>(s, tmem, args.timeout_ns);
}

// Input staging of one layer, one block of 1024 threads per token:
//   norm_w == NULL: act[t] = fp32(x[t]) (x bf16), and resid[t] = act[t] when resid != NULL;
//   norm_w != NULL: act[t] = resid[t] * w / sqrt(mean(resid[t]^2) + eps)  (RMSNorm);
// then the expert operand of act[t]: 8 E2M1 terms per MX block (xb4, xsf).
constexpr int kPrepThreads = 1024;
__global__ void __launch_bounds__(kPrepThreads) prep_layer_kernel(const __nv_bfloat16* __restrict__ x, int T, int H,
                                                                  float* resid, const __nv_bfloat16* __restrict__ norm_w,
                                                                  float eps, float* __restrict__ act,
                                                                  uint8_t* __restrict__ xb4, uint8_t* __restrict__ xsf) {
    __shared__ float red[32];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kPer = 16;   // H <= 16384: at most 16 values per thread
    float v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int h = threadIdx.x + i * kPrepThreads;
        v[i] = 0.0f;
        if (h < H) v[i] = norm_w ? resid[(size_t)t * H + h] : __bfloat162float(x[(size_t)t * H + h]);
    }
    if (norm_w) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.0f;
        for (int i = 0; i < 32; ++i) tot += red[i];
        const float inv = 1.0f / sqrtf(tot / (float)H + eps);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int h = threadIdx.x + i * kPrepThreads;
            if (h < H) v[i] = v[i] * inv * __bfloat162float(norm_w[h]);
        }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int h = threadIdx.x + i * kPrepThreads;   // block (h / 32) = 32 i + warp, element lane
        if (i * kPrepThreads < H) {                      // warp-uniform (H is a multiple of 1024 or the tail is whole blocks)
            if (h < H) {
                act[(size_t)t * H + h] = v[i];
                if (resid && !norm_w) resid[(size_t)t * H + h] = v[i];
            }
            if (h - lane < H) {
                uint32_t sb0, sb1;
                const uint32_t codes = split_e2m1_terms(v[i], sb0, sb1);
                store_act_terms(xb4, xsf, H, t, h / 32, lane, codes, sb0, sb1);
            }
        }
    }
}

}  // namespace moe
