"""Oracle for the MXFP4 MoE expert layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 CPU statement of what one MoE layer of a speculative
verify block computes.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the product (the CUDA library and its Python
binding) never does and shares no code with it.

Sources, by page title and section:

* "MiMo x TileRT" (page 1), section "第一层：FP4 选择性量化": expert weights are
  stored in the OCP Microscaling FP4 format (MXFP4); the router keeps higher
  precision.  Section "万亿参数推理为什么特别难": decode tokens/s is bounded by
  memory bandwidth divided by the bytes read per token.
* "MiMo 把 1T 模型推到每秒千 token" (page 3), section "FP4：只量化 MoE expert":
  weights are split into small blocks that share one scale, elements are FP4;
  the router's top-k choice is precision-sensitive.  Section "DFlash": one
  target forward verifies the 8 drafted positions at once.
* The implementation guide (page 5), "关键实现细节" item 1: the expert linears
  are gate_proj / up_proj / down_proj; the worked bandwidth bound numbers.
* The OCP Microscaling Formats v1.0 definition that pages 1 and 5 cite as a
  source: FP4 E2M1 elements (1 sign, 2 exponent bits with bias 1, 1 mantissa
  bit, no Inf/NaN), E8M0 block scales (2^(b-127), 0xFF = NaN), block size 32,
  and the conversion rule X = 2^(floor(log2(amax)) - emax_elem) with
  emax_elem = 2 for E2M1, elements rounded to nearest-even and saturated.

Readings taken where the pages are silent:
* SwiGLU expert: a = silu(Wg x) * (Wu x), d = Wd a.
* Gates are the softmax over the k selected logits; the router bias is part
  of the logits (selection and gates).
* Top-k orders by (logit descending, expert index ascending).
* Inside one expert, tokens are listed ascending by (token, slot).
* Nibble 2j of a row is the low nibble of byte j; matrices are [out, in]
  row-major with the contraction dimension contiguous; scales are
  [out, in / 32].
* RMSNorm n = r * w / sqrt(mean(r^2) + eps); a layer of the stack is
  r <- r + MoE(RMSNorm(r)).

Every pin of this file lives in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

MX_BLOCK = 32


# --------------------------------------------------------------------------- format


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP MX v1.0 FP4 element definition).

    bit 3 = sign, bits 2..1 = exponent (bias 1), bit 0 = mantissa.
    Exponent field 0 is subnormal: 0.5 * m.  Otherwise 2^(e-1) * (1 + m/2).
    """
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


E2M1_VALUES = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e8m0_value(b: np.ndarray) -> np.ndarray:
    """Scale of an E8M0 byte: 2^(b - 127); 0xFF is NaN (OCP MX v1.0)."""
    b = np.asarray(b, dtype=np.int64)
    out = np.ldexp(1.0, b - 127).astype(np.float64)
    return np.where(b == 255, np.nan, out)


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """uint8 [..., n/2] -> codes [..., n]; element 2j is the low nibble of byte j."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0x0F
    out[..., 1::2] = q >> 4
    return out


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """W[r, c] = e2m1(nibble(r, c)) * 2^(S[r, c/32] - 127), in fp64."""
    codes = unpack_nibbles(q)
    rows, cols = codes.shape
    assert s.shape == (rows, cols // MX_BLOCK), (s.shape, codes.shape)
    if np.any(np.asarray(s) == 255):
        raise ValueError("E8M0 scale byte 0xFF (NaN) in input")
    scale = np.repeat(e8m0_value(s), MX_BLOCK, axis=1)
    return E2M1_VALUES[codes] * scale


def _round_e2m1_magnitude(v: np.ndarray) -> np.ndarray:
    """|v| (fp64, >= 0) -> magnitude code 0..7: nearest grid point, ties to the
    even code, saturating at 6 (the largest E2M1 magnitude)."""
    grid = E2M1_VALUES[:8]
    v = np.minimum(v, grid[-1])
    hi = np.clip(np.searchsorted(grid, v, side="left"), 1, 7)  # grid[hi-1] < v <= grid[hi] (or v == 0)
    lo = hi - 1
    d_lo = v - grid[lo]
    d_hi = grid[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


def quantize(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 [rows, cols] -> (nibbles uint8 [rows, cols/2], scales uint8 [rows, cols/32]).

    Per 32-element block: amax = max |w|; the shared scale is
    X = 2^(floor(log2 amax) - 2) (2 = exponent of the largest E2M1 value, 6),
    stored as the E8M0 byte floor(log2 amax) - 2 + 127 clamped to [0, 254];
    an all-zero block takes byte 127.  Each element w / X is rounded to the
    nearest E2M1 value, ties to even, saturating at +-6; the sign bit is the
    sign of w (so -0.0 and small negatives that round to zero keep it).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % MX_BLOCK == 0
    blocks = w.reshape(rows, cols // MX_BLOCK, MX_BLOCK).astype(np.float64)
    amax = np.fabs(blocks).max(axis=2)
    _, ex = np.frexp(amax)                       # amax = m * 2^ex, m in [0.5, 1)
    byte = np.clip(ex - 1 - 2 + 127, 0, 254)
    byte = np.where(amax == 0, 127, byte).astype(np.int64)
    v = blocks / np.ldexp(1.0, byte - 127)[..., None]
    mag = _round_e2m1_magnitude(np.fabs(v))
    sign = np.signbit(blocks).astype(np.uint8)
    codes = (sign << 3 | mag).reshape(rows, cols)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return q, byte.astype(np.uint8)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- routing


def router_logits(x: np.ndarray, wr: np.ndarray, b: np.ndarray | None) -> np.ndarray:
    """logit[t, e] = sum_h x[t, h] * Wr[e, h] + b[e], in fp64."""
    z = np.asarray(x, np.float64) @ np.asarray(wr, np.float64).T
    if b is not None:
        z = z + np.asarray(b, np.float64)[None, :]
    return z


def topk_gates(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k by (logit desc, expert asc); gates = softmax over the k chosen logits."""
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))  # last key is primary
        sel = order[:k]
        idx[t] = sel
        z = logits[t, sel]
        ez = np.exp(z - z[0])
        gate[t] = ez / ez.sum()
    return idx, gate


def assignment(idx: np.ndarray, E: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Token-to-expert grouping of the (token, slot) pairs.

    counts[e] = number of pairs routed to e; offsets = exclusive prefix sum
    (length E+1); perm lists the pair ids t*k + j grouped by expert, ascending
    by (t, j) inside an expert.
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int32)
    for e in idx.reshape(-1):
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.empty(T * k, dtype=np.int32)
    fill = offsets[:-1].copy()
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            perm[fill[e]] = t * k + j
            fill[e] += 1
    return counts, offsets, perm


# --------------------------------------------------------------------------- experts


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


class ExpertMatrices:
    """Dequantised fp64 matrices of one expert (gate, up [I, H]; down [H, I])."""

    def __init__(self, gate_q, gate_s, up_q, up_s, down_q, down_s):
        self.gate = dequant(gate_q, gate_s)
        self.up = dequant(up_q, up_s)
        self.down = dequant(down_q, down_s)

    def ffn(self, xrow: np.ndarray) -> np.ndarray:
        """SwiGLU expert: Wd (silu(Wg x) * (Wu x))."""
        gv = self.gate @ xrow
        uv = self.up @ xrow
        return self.down @ (silu(gv) * uv)


def moe_layer(x: np.ndarray, wr, b, k: int, expert_fn) -> dict:
    """One MoE layer on a verify block.

    x: fp64 [T, H]; wr: fp64 [E, H]; b: fp64 [E] or None;
    expert_fn(e) -> ExpertMatrices (called once per distinct routed expert).
    Returns the routing, the assignment and y[t] = sum_j gate[t, j] * FFN_{idx[t, j]}(x_t),
    summed in slot order j = 0..k-1.
    """
    T = x.shape[0]
    E = wr.shape[0]
    logits = router_logits(x, wr, b)
    idx, gate = topk_gates(logits, k)
    counts, offsets, perm = assignment(idx, E)
    d = {}
    for e in np.nonzero(counts)[0]:
        m = expert_fn(int(e))
        for p in perm[offsets[e]:offsets[e + 1]]:
            t, j = divmod(int(p), k)
            d[(t, j)] = m.ffn(x[t])
    y = np.zeros_like(x, dtype=np.float64)
    for t in range(T):
        for j in range(k):
            y[t] += gate[t, j] * d[(t, j)]
    return dict(logits=logits, idx=idx, gate=gate, counts=counts, offsets=offsets, perm=perm, y=y)


def moe_token(xrow: np.ndarray, wr, b, k: int, expert_fn) -> dict:
    """The layer's output for one token alone (the layer is per token)."""
    r = moe_layer(xrow[None, :], wr, b, k, expert_fn)
    return dict(idx=r["idx"][0], gate=r["gate"][0], logits=r["logits"][0], y=r["y"][0])


def rmsnorm(r: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """n = r * w / sqrt(mean_h(r^2) + eps), per row, fp64."""
    r = np.asarray(r, np.float64)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    return r * np.asarray(w, np.float64) / np.sqrt(ms + eps)


def moe_stack(x: np.ndarray, layers: list, k: int, eps: float) -> dict:
    """L consecutive pre-norm MoE layers with residual: r <- r + MoE_l(RMSNorm_l(r)).

    layers[l] = dict(wr, b, norm_w, expert_fn).  Returns the final residual and
    each layer's routing.
    """
    r = np.asarray(x, np.float64).copy()
    per_layer = []
    for L in layers:
        n = rmsnorm(r, L["norm_w"], eps)
        out = moe_layer(n, L["wr"], L["b"], k, L["expert_fn"])
        r = r + out["y"]
        per_layer.append(out)
    return dict(y=r, layers=per_layer)


# --------------------------------------------------------------------------- metric


def implied_tokens_per_s(bandwidth_bytes_per_s: float, bytes_per_token: float) -> float:
    """Memory-bound decode bound: tokens/s <= bandwidth / bytes read per token
    (page 1 "万亿参数推理为什么特别难"; page 5 "关键实现细节" item 1)."""
    return bandwidth_bytes_per_s / bytes_per_token


def verify_tokens_per_s(seconds_per_verify: float, acceptance_length: float = 6.30) -> float:
    """Decode tokens/s when each verify forward of the 8-position block yields
    `acceptance_length` accepted tokens (coding average 6.30, page 3 "DFlash")."""
    return acceptance_length / seconds_per_verify


def topk_margin(logits_row: np.ndarray, k: int) -> float:
    """Smallest gap between adjacent logits among the top-(k+1) of one token."""
    top = np.sort(np.asarray(logits_row, np.float64))[::-1][: min(k + 1, logits_row.size)]
    return float(np.min(top[:-1] - top[1:])) if top.size > 1 else math.inf


def accept_block(logits: np.ndarray, tokens: np.ndarray) -> dict:
    """Acceptance of verify blocks ("MiMo 把 1T 模型推到每秒千 token", DFlash section: the
    target scores all drafted positions in one forward and the longest agreeing prefix
    is kept).  logits [S, B, V] (position i predicts the token of position i + 1);
    tokens [S, B] (position 0 the last committed token, 1..B-1 the drafts).  Per
    stream: target = greedy token per position (first maximum; NaN as -inf); a = number
    of leading drafts equal to the target's prediction for their position; accepted =
    a + 1 tokens yielded; next_token = target[a]."""
    lg = np.where(np.isnan(logits), -np.inf, logits)
    target = np.argmax(lg, axis=2).astype(np.int32)   # numpy returns the first maximum
    S, B = tokens.shape
    accepted = np.zeros(S, dtype=np.int32)
    nxt = np.zeros(S, dtype=np.int32)
    for s in range(S):
        a = 0
        while a + 1 < B and tokens[s, a + 1] == target[s, a]:
            a += 1
        accepted[s] = a + 1
        nxt[s] = target[s, a]
    return dict(target=target, accepted=accepted, next_token=nxt)
