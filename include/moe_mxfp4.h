/*
 * moe_mxfp4.h -- C ABI of the MXFP4 Mixture-of-Experts expert layer for GB300 (sm_103a).
 *
 * One call runs one MoE layer (or a stack of pre-norm MoE layers) over a
 * speculative-decoding verify block: router GEMM, softmax over the top-k
 * logits, token-to-expert grouping, per-expert SwiGLU FFN on MXFP4 weights
 * that are dequantised in registers, and the gate-weighted combine.
 *
 * Where the operation comes from (page title, section):
 *  - "MiMo x TileRT" (blog.hypho.cn), "第一层：FP4 选择性量化": only the MoE
 *    expert weights are stored in OCP Microscaling FP4 (MXFP4); the router keeps
 *    higher precision.  "万亿参数推理为什么特别难": decode speed is bounded by
 *    HBM bandwidth / bytes read per token, so the layer is judged on bytes moved.
 *  - "MiMo 把 1T 模型推到每秒千 token" (vatt-ghern), "FP4：只量化 MoE expert":
 *    blocks of weights share one scale, elements are FP4; the router's top-k is
 *    precision-sensitive.  "DFlash：block-level masked 並行草稿": one target
 *    forward verifies 8 drafted positions.  "persistent engine kernel 與 warp
 *    specialization": one resident launch instead of one launch per operator.
 *  - Implementation guide (shengyayun), "关键实现细节" items 1 and 3: expert
 *    linears gate_proj / up_proj / down_proj; per-launch gaps of 5-10 us.
 *  - OCP Microscaling Formats v1.0 (cited by the pages): E2M1 elements, E8M0
 *    scales 2^(b-127) with 0xFF = NaN, 32 elements per scale.
 *
 * Conventions
 *  - Every pointer named *_dev is a device pointer owned by the caller; the
 *    library never allocates device memory (the caller provides a workspace
 *    whose size moe_mxfp4_workspace_bytes reports) and never frees caller memory.
 *  - Weights are BORROWED at create time: they must stay allocated and unchanged
 *    until moe_mxfp4_destroy.  create makes no copy or repack (moe_mxfp4_pack, below,
 *    is a separate call the caller makes once, into memory it owns).
 *  - Calls are asynchronous on the given stream (a cudaStream_t passed as void*,
 *    NULL = legacy default stream) unless stated otherwise.  Errors the host can
 *    see are returned at once; errors found on the device (a NaN scale byte, a
 *    device wait that timed out, a workspace whose state section was overwritten)
 *    are written to a status word in the workspace and returned by moe_mxfp4_check.
 *    In the persistent forward (the default) such an error stays there: later
 *    forwards on that workspace do nothing until moe_mxfp4_check (or
 *    moe_mxfp4_forward_host, or moe_mxfp4_forward_static) reads it, which also
 *    returns the workspace's state section to rest.  The per-phase paths
 *    (MOE_FLAG_MULTI_KERNEL) clear the status words at the start of each forward.
 *    No call aborts or throws.
 *  - One handle + one workspace may be used by one stream at a time.
 *
 * Layouts (row-major, contraction dimension contiguous):
 *  - x: bf16 [T, H].   y: fp32 [T, H] (bf16 with MOE_FLAG_OUT_BF16).
 *  - router_w: bf16 [E, H];  router_b: fp32 [E] (may be NULL = zero).
 *  - gate_q, up_q: uint8 [E, I, H/2];  gate_s, up_s: uint8 [E, I, H/32].
 *  - down_q: uint8 [E, H, I/2];        down_s: uint8 [E, H, I/32].
 *    Element 2j of a row is the LOW nibble of byte j; a nibble is an E2M1 code
 *    (bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa).  Scale byte
 *    S[r, c/32] multiplies elements c of row r by 2^(S - 127).
 *  - norm_w: bf16 [H] (required with MOE_FLAG_NORM).
 *  Every base pointer must be 16-byte aligned; H and I must be multiples of 128.
 *  - packed (optional, see moe_mxfp4_pack): the same expert bytes rearranged
 *    tile-major, so that the expert kernels read every stage of weights as one
 *    contiguous run of memory.  Requires H and I multiples of 512.
 *
 * What a layer computes (per token t):
 *   logit[e] = sum_h x[t,h] Wr[e,h] + b[e]
 *   (idx, gate) = top-k by (logit desc, expert asc); gate = softmax(selected logits)
 *   for slot j: e = idx[j]; a = silu(Wg_e x_t) * (Wu_e x_t); d_j = Wd_e a
 *   y[t] = sum_j gate[j] d_j  (slot order j = 0..k-1)
 * With MOE_FLAG_NORM the call runs num_layers layers r <- r + MoE_l(RMSNorm_l(r))
 * with RMSNorm(r) = r * w / sqrt(mean(r^2) + eps), r_0 = x, and y = r_L.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define MOE_OK               0
#define MOE_ERR_INVALID_ARG (-1) /* bad size, NULL or misaligned pointer, T > max_tokens */
#define MOE_ERR_UNSUPPORTED (-2) /* no sm_103 device current, or a shape outside the limits */
#define MOE_ERR_CUDA        (-3) /* a CUDA runtime call failed */
#define MOE_ERR_TIMEOUT     (-4) /* a device-side wait gave up (grid barrier / expert counter) */
#define MOE_ERR_BAD_SCALE   (-5) /* an E8M0 scale byte of a routed expert is 0xFF (NaN) */
#define MOE_ERR_WORKSPACE   (-6) /* workspace NULL, misaligned (256 B) or too small; on the device:
                                      its state section was overwritten between forwards */

/* ---- config flags ------------------------------------------------------- */
#define MOE_FLAG_NORM         (1u << 0) /* pre-norm residual stack (see above) */
#define MOE_FLAG_OUT_BF16     (1u << 1) /* y is bf16 instead of fp32 */
#define MOE_FLAG_MULTI_KERNEL (1u << 2) /* one launch per phase (comparison path) */
#define MOE_FLAG_NO_DENSE     (1u << 3) /* blocks routed through the workspace (T*k > 64 or T*E > 8192) use
                                          * chunks of 16 pairs x 8 E2M1 terms per activation instead of the
                                          * dense operand of 32 pairs x 4 terms (see moe_mxfp4_forward) */
#define MOE_FLAG_DEBUG_STALL  (1u << 4) /* testing aid: the forward withholds one device-side signal (one
                                          * CTA's first grid-barrier arrival in the persistent forward; the
                                          * gate/up completions of the first routed expert in the one-launch-
                                          * per-phase forward), so its waits run out after timeout_us and the
                                          * status becomes MOE_ERR_TIMEOUT; nothing hangs or faults */
#define MOE_FLAG_TRACE        (1u << 5) /* profiling aid: the expert phase of the first layer records the
                                          * first CTA's per-stage timestamps in the workspace (below) */

typedef struct moe_mxfp4_handle moe_mxfp4_handle; /* opaque, host-side */

typedef struct {
    int32_t num_layers;   /* >= 1; > 1 requires MOE_FLAG_NORM */
    int32_t hidden;       /* H, multiple of 128, <= 16384 */
    int32_t inter;        /* I, multiple of 128, <= 16384 */
    int32_t num_experts;  /* E, 1..1024 */
    int32_t top_k;        /* k, 1..min(E, 32) */
    int32_t max_tokens;   /* largest T a forward will get, 1..4096 */
    float rms_eps;        /* RMSNorm epsilon (used with MOE_FLAG_NORM) */
    uint32_t flags;       /* MOE_FLAG_* */
    int32_t expert_begin; /* experts [expert_begin, expert_end) are computed here; */
    int32_t expert_end;   /* tokens routed elsewhere contribute 0 (expert-parallel shard). 0,0 = all */
    int32_t timeout_us;   /* bound of every device-side wait in microseconds; 0 = default (200000) */
} moe_mxfp4_config;

typedef struct {
    const void* router_w_dev;   /* bf16 [E, H] */
    const float* router_b_dev;  /* fp32 [E] or NULL */
    const uint8_t* gate_q_dev;  /* [E, I, H/2] */
    const uint8_t* gate_s_dev;  /* [E, I, H/32] */
    const uint8_t* up_q_dev;    /* [E, I, H/2] */
    const uint8_t* up_s_dev;    /* [E, I, H/32] */
    const uint8_t* down_q_dev;  /* [E, H, I/2] */
    const uint8_t* down_s_dev;  /* [E, H, I/32] */
    const void* norm_w_dev;     /* bf16 [H] or NULL */
    const uint8_t* packed_dev;  /* NULL, or this layer's experts in the packed layout (moe_mxfp4_pack,
                                 * 256-byte aligned): the forward then reads the experts from here only
                                 * and gate_q_dev .. down_s_dev may be NULL */
} moe_mxfp4_layer;

/* Optional copies of the routing of every layer, written by a forward when the
 * pointers are non-NULL (device memory, caller-owned):
 *   topk_idx int32 [L, T, k], topk_gate fp32 [L, T, k], expert_counts int32 [L, E],
 *   expert_offsets int32 [L, E+1], perm int32 [L, T*k] (pair ids t*k+j grouped by
 *   expert, ascending by (t, j) inside an expert).
 * expert_events, when non-NULL, points to 2*L cudaEvent_t handles (host array,
 * caller-created): the forward records events[2l] on the stream right before the
 * expert kernel of layer l and events[2l+1] right after it, so a caller can time
 * that kernel alone. */
typedef struct {
    int32_t* topk_idx_dev;
    float* topk_gate_dev;
    int32_t* expert_counts_dev;
    int32_t* expert_offsets_dev;
    int32_t* perm_dev;
    void* const* expert_events;
} moe_mxfp4_debug;

/* Validates the config and the layer pointers (alignment, device), and checks
 * that the current device is an sm_103 GPU.  layers points to num_layers
 * descriptors (host memory, copied).  On success *out receives a handle. */
int moe_mxfp4_create(const moe_mxfp4_config* cfg, const moe_mxfp4_layer* layers,
                     moe_mxfp4_handle** out);

/* Bytes of device workspace a forward over num_tokens tokens needs.  The first 512
 * bytes hold the status words (code at 0, detail at 4), the grid-barrier word (16), the
 * routing flag (20), the abort flag (24) and the state tag (32, uint64); in a persistent
 * forward, bytes 64..511 receive CTA 0's
 * %globaltimer (uint64 ns) at the end of each phase (entry i at 64 + 8 i: start,
 * input staging, and per layer l < 8: router 2+4l, routing 3+4l, experts 4+4l, combine
 * 5+4l; for the first layer also the routing sub-steps at 34..38 (blocks routed through
 * the workspace) or 40..44, the steps of router unit 0 at 48..52 (unit 1 when the block
 * has several token blocks), the end of CTA 0's router units at 53 and of its operand
 * split at 54), for profiling, and
 * bytes 512..2559 receive each CTA's %globaltimer when it finished (CTA i at 512 + 8 i).
 * With MOE_FLAG_TRACE, bytes 4096..16383 receive the first layer's expert-phase
 * timestamps of CTA 0 as 6 arrays of 256 uint64 (ns, ring stage or item i < 256):
 * producer issues stage i, scale-factor warp sees it land, scale factors written,
 * MMA thread starts it, MMAs issued, epilogue starts item i. */
int moe_mxfp4_workspace_bytes(const moe_mxfp4_handle* h, int32_t num_tokens, size_t* bytes);

/* Runs the layer (stack) on num_tokens rows of x_dev into y_dev.  workspace_dev
 * must be 256-byte aligned and at least moe_mxfp4_workspace_bytes long; its
 * contents need no initialisation.  The persistent forward keeps a state section at
 * the start of the workspace (16 KB of status words, then the counters of its work
 * queues; the same bytes for every num_tokens) between forwards: each launch leaves it
 * at rest, so the forward is one kernel launch with no clearing copy before it.  The
 * library zeroes the section (one small extra launch) the first time this handle's
 * persistent forward meets the workspace, after another handle or a per-phase forward
 * used it, and after an error was read from it.  Between forwards the caller leaves
 * the section's bytes alone; if something else wrote them, the forward finds a wrong
 * state tag, records MOE_ERR_WORKSPACE and does nothing.  x_dev and y_dev may not
 * alias each other or the workspace.  num_tokens == 0 is a no-op.  dbg may be NULL.
 * Arithmetic: the router's products of x are exact and summed in fp32; in a residual
 * stack, RMSNorm(r) = (r * w_norm) / rms(r) with one factor 1 / rms(r) per token, so the
 * router sums the fp32 products of y = r * w_norm (fp32) with its bf16 weights per
 * 256-column block, in block order, and scales the sum by the factor, and the experts
 * take y as their input and scale their gate/up outputs by it; each expert weight
 * is its exact MXFP4 value; each activation (the layer input, and h = silu(g) * u)
 * enters the tensor cores as a sum of E2M1 terms with per-32 E8M0 scales, each term
 * encoding the residual of the previous ones.  A block of at most 64 (token, slot)
 * pairs (T*k <= 64, T*E <= 8192) works through chunks of at most 8 pairs of an expert
 * with 8 terms per activation (for N(0,1) inputs the sum stays within ~1e-7 of the
 * 32-block's maximum); larger blocks use chunks of up to 32 pairs with 4 terms (within
 * ~3e-4 of the block maximum; each weight tile then serves four times the pairs), or
 * of up to 16 pairs with 8 terms when MOE_FLAG_NO_DENSE is set.  Products are summed
 * in fp32. */
int moe_mxfp4_forward(moe_mxfp4_handle* h, const void* x_dev, int32_t num_tokens, void* y_dev,
                      void* workspace_dev, size_t workspace_bytes, void* stream,
                      const moe_mxfp4_debug* dbg);

/* The same forward on HOST buffers: copies x_host (bf16 [T, H]) into the
 * workspace, runs the forward, copies y back to y_host (fp32 or bf16 [T, H])
 * and synchronises the stream once (the status words are copied behind y on the
 * same stream into a 64-byte pinned buffer that the handle allocates on first use
 * and frees in moe_mxfp4_destroy).  Pinned host memory makes the copies of x and y
 * asynchronous.  Calls on one handle from several threads are serialised from the
 * status copy on.  Returns the device status (as moe_mxfp4_check), or MOE_ERR_CUDA
 * when a copy, the pinned allocation or the synchronisation fails. */
int moe_mxfp4_forward_host(moe_mxfp4_handle* h, const void* x_host, int32_t num_tokens, void* y_host,
                           void* workspace_dev, size_t workspace_bytes, void* stream);

/* Synchronises the stream and returns the device status word of this workspace: the
 * first error a persistent forward recorded since the status was last read, or the
 * last per-phase forward's status (MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_BAD_SCALE or
 * MOE_ERR_WORKSPACE).  After an error it returns the state section to rest, so the
 * next forward runs normally. */
int moe_mxfp4_check(moe_mxfp4_handle* h, const void* workspace_dev, void* stream);

/* Frees the handle (its host memory, including the pinned status buffer of
 * moe_mxfp4_forward_host).  NULL is ignored. */
void moe_mxfp4_destroy(moe_mxfp4_handle* h);

/* Static description of a status code. */
const char* moe_mxfp4_status_string(int status);

/* Allocation-free forward.  The pages have no counterpart to this call; it exists for
 * callers that cannot allocate device memory at the point where they run the layer --
 * for example a host program that reserved all of HBM up front for its own pool, a
 * plugin inside a framework that owns every device allocation, or a latency-bound loop
 * that cannot afford cudaMalloc's device-wide synchronisation.
 * It runs exactly moe_mxfp4_forward, but its workspace is a fixed static array inside
 * this library (MOE_MXFP4_STATIC_WORKSPACE_BYTES = 16 MiB per GPU, held from the moment
 * the library's device code is loaded until the process exits) instead of caller memory.
 * The caller still provides x_dev and y_dev (device memory, as for moe_mxfp4_forward).
 *  - Returns MOE_ERR_WORKSPACE, and runs nothing, when num_tokens needs more workspace
 *    than the static array holds (moe_mxfp4_workspace_bytes tells the need).
 *  - The first call on a device, with that device current, looks up the array's device
 *    address (once per device); make that first call before any stream capture.  The
 *    address is kept for the life of the process: after cudaDeviceReset on a device, do
 *    not call this function again on that device.
 *  - All calls on a device share the one array and leave their contents in it; the
 *    forward re-initialises everything it needs.  Calls whose work overlaps on the GPU
 *    (different streams, or different handles at the same time) race on the array.
 *  - Never calls cudaMalloc, cudaFree or any other allocating routine.
 *  - Synchronises the stream before it returns and returns the device status of the
 *    call (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_BAD_SCALE), like moe_mxfp4_check. */
#define MOE_MXFP4_STATIC_WORKSPACE_BYTES (16u << 20)
int moe_mxfp4_forward_static(moe_mxfp4_handle* h, const void* x_dev, int32_t num_tokens, void* y_dev,
                             void* stream);

/* Packed expert layout.  The canonical layout above stores each matrix row by row, so
 * the weights the kernels stream per 256-K stage of a work item (the gate and the up
 * rows of a 128-row block, or 256 down rows: 32 KB of codes) are 256 runs of 128 bytes
 * in one or two matrices, and the scales of a few consecutive 32-blocks are a few bytes
 * per row: each stage costs two or four copy requests through two tensor maps.  The
 * packed layout holds the same bytes, rearranged once (when the weights are loaded,
 * like any inference engine's weight preprocessing), so that each stage and each scale
 * group is one contiguous run read by one copy ("MiMo x TileRT", 万亿参数推理为什么特别难:
 * decode speed is HBM bandwidth over bytes read, so the bytes must arrive at the full
 * rate).  Three 256-byte-aligned sections:
 *   codes:     gate/up tiles [E][I/128][H/256][256 rows: 128 gate, then the same 128 up][128 B],
 *              then down tiles [E][H/256][I/256][256 rows][128 B]
 *   scales_gu: [E][I/128][H/256/G_H][256 rows: 128 gate, 128 up][8 G_H B]
 *   scales_d:  [E][H/256][I/256/G_I][256 rows][8 G_I B]
 * where rows are in order within a tile, a code row holds the 128 bytes of its matrix
 * row at K offset 256 st, and G_K (256-K stages per scale group) is the largest of 8, 6,
 * 4, 2 that divides K/256.  The packed buffer has exactly the bytes of the canonical one
 * plus section padding.  moe_mxfp4_packed_bytes reports its size for (H, I, E);
 * moe_mxfp4_pack fills it from a layer's canonical pointers (device memory,
 * caller-owned; asynchronous on stream; the source must stay unchanged until the copy
 * has run).  Both return MOE_ERR_UNSUPPORTED when H or I is not a multiple of 512,
 * MOE_ERR_INVALID_ARG for a bad size or pointer (packed_dev must be 256-byte aligned and
 * packed_bytes at least the reported size). */
int moe_mxfp4_packed_bytes(int32_t hidden, int32_t inter, int32_t num_experts, size_t* bytes);
int moe_mxfp4_pack(int32_t hidden, int32_t inter, int32_t num_experts, const moe_mxfp4_layer* layer,
                   void* packed_dev, size_t packed_bytes, void* stream);

/* The activation encoding of the expert kernels, on its own (see moe_mxfp4_forward's
 * arithmetic note): each fp32 value of a 32-element block becomes the sum of E2M1 terms
 * with one E8M0 scale per term and block.  Term j has scale X_j = 2^(floor(log2 m_j) - 2),
 * doubled when m_j > 6 X_j, where m_j is the largest magnitude of the block's residual
 * after terms 0..j-1; its codes round residual / X_j to the nearest E2M1 value (ties to
 * the even code); a residual below 2^-119 ends the sum (its terms are code 0, scale byte
 * 0).  Each term at least quarters the block's largest residual, so the first t terms
 * are within 4^-t of the block's largest magnitude (the kernels use t = 8, or t = 4 for
 * the dense operand of larger blocks).  x_dev: fp32 [n_blocks, 32]; codes_dev: uint32
 * [n_blocks, 32] (element i: term j's code in bits 4j..4j+3, 8 terms); scales_dev: uint8
 * [n_blocks, 8] (term j's E8M0 byte).  Device pointers, asynchronous on stream; NaN
 * inputs are not supported.  MOE_ERR_INVALID_ARG for n_blocks < 0 or a NULL pointer. */
int moe_mxfp4_split_terms(const float* x_dev, int64_t n_blocks, uint32_t* codes_dev, uint8_t* scales_dev,
                          void* stream);

/* MXFP4 conversion of an fp32 matrix w_dev [rows, cols] (cols a multiple of 32)
 * into nibbles q_dev [rows, cols/2] and E8M0 scales s_dev [rows, cols/32], by the
 * OCP MX v1.0 rule: per block of 32, X = 2^(floor(log2 amax) - 2) (byte clamped to
 * [0, 254]; an all-zero block gets byte 127); elements w/X rounded to the nearest
 * E2M1 value, ties to even, saturating at +-6; the sign bit is the sign of w.
 * NaN inputs are not supported.  Device pointers (w_dev and q_dev 16-byte
 * aligned), asynchronous on stream. */
int moe_mxfp4_quantize(const float* w_dev, int64_t rows, int64_t cols, uint8_t* q_dev, uint8_t* s_dev,
                       void* stream);

/* Acceptance of speculative verify blocks ("MiMo 把 1T 模型推到每秒千 token", DFlash
 * section: one target forward scores the drafted positions of a block; the longest
 * prefix the target agrees with is kept and the rest discarded).  Block position i of
 * stream s holds input token tokens[s, i] (position 0: the last committed token,
 * positions 1..B-1: drafted tokens), and the target's logits at position i predict
 * the token of position i + 1.  The call computes, per stream:
 *   target[s, i]   = argmax_v logits[s, i, v]   (lowest index among equal maxima; NaN
 *                    ranks as -inf)
 *   a              = the largest m <= B-1 with tokens[s, i] == target[s, i-1], i = 1..m
 *   accepted[s]    = a + 1   (tokens this verify yields: the a accepted drafts and the
 *                    target's own next token; the pages' "acceptance length")
 *   next_token[s]  = target[s, a]
 * logits_dev: fp32 [S, B, V]; tokens_dev: int32 [S, B]; target_dev: int32 [S, B]
 * (output, also the working array); accepted_dev, next_token_dev: int32 [S] (outputs;
 * next_token_dev may be NULL).  Device pointers, caller-owned; asynchronous on stream.
 * MOE_ERR_INVALID_ARG for S < 0, B < 1, V < 1, S*B or V above 2^31 - 1, or a NULL
 * required pointer; S = 0 is a no-op. */
int moe_mxfp4_accept(const float* logits_dev, const int32_t* tokens_dev, int32_t num_streams, int32_t block,
                     int64_t vocab, int32_t* target_dev, int32_t* accepted_dev, int32_t* next_token_dev,
                     void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXFP4_H */
