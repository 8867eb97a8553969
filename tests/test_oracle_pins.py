"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible mistake in the oracle (a wrong
exponent bias, swapped nibble order, wrong scale index, a dropped sign, a
transposed operand, a wrong tie rule, a missing gate or residual term) fails
it.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------------------- format


def test_e2m1_decode_matches_format_table():
    table = {int(c): float(v) for c, v in _golden_rows("e2m1_table.txt")}
    assert len(table) == 16
    for c in range(16):
        assert O.E2M1_VALUES[c] == table[c], c
        assert math.copysign(1.0, O.E2M1_VALUES[c]) == math.copysign(1.0, table[c]), c


def test_e8m0_scale_values():
    b = np.array([0, 1, 126, 127, 128, 200, 254])
    got = O.e8m0_value(b)
    want = [2.0 ** (int(v) - 127) for v in b]
    assert list(got) == want
    assert np.isnan(O.e8m0_value(np.array([255]))[0])


def test_dequant_nibble_order_and_scale_index():
    # one row of 64 elements: byte 0 = 0x21 -> element 0 = code 1 (0.5), element 1 = code 2 (1.0)
    q = np.zeros((1, 32), np.uint8)
    q[0, 0] = 0x21
    q[0, 16] = 0xF7           # element 32 = code 7 (6.0), element 33 = code 15 (-6.0)
    s = np.array([[127, 129]], np.uint8)   # block 1 scaled by 4
    w = O.dequant(q, s)
    assert w[0, 0] == 0.5 and w[0, 1] == 1.0
    assert w[0, 32] == 24.0 and w[0, 33] == -24.0
    assert np.count_nonzero(w) == 4


def test_dequant_rejects_nan_scale():
    with pytest.raises(ValueError):
        O.dequant(np.zeros((1, 16), np.uint8), np.array([[255]], np.uint8))


def test_bf16_bits_exact():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x3E00], np.uint16)
    got = O.bf16_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0
    assert got[2] == 2.0 ** -133
    assert got[3] == (2 - 2 ** -7) * 2.0 ** 127
    assert got[4] == 0.125


# ----------------------------------------------------------------------------- quantizer


def _block_with_scale_anchor(values, anchor=7.96875):
    """Blocks of 32 whose first element fixes floor(log2 amax) = 2 (scale 2^0)."""
    n = len(values)
    nb = -(-n // 31)
    pad = np.zeros(nb * 31, np.float32)
    pad[:n] = values
    blocks = np.concatenate([np.full((nb, 1), anchor, np.float32), pad.reshape(nb, 31)], axis=1)
    return blocks.reshape(1, -1), nb


def _brute_force_code(v: float) -> int:
    """Nearest E2M1 magnitude by exhaustive search; ties -> even code; saturate."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = min(abs(v), 6.0)
    best = None
    for c, g in enumerate(grid):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1] | (8 if math.copysign(1.0, v) < 0 else 0)


def test_quantize_ties_to_even():
    # midpoints of the E2M1 grid and the code round-to-nearest-even picks
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    vals = np.array(list(ties) + [-v for v in ties], np.float32)
    w, nb = _block_with_scale_anchor(vals)
    q, s = O.quantize(w)
    assert np.all(s == 127)
    deq = O.dequant(q, s).reshape(nb, 32)[:, 1:].reshape(-1)[: len(vals)]
    want = list(ties.values()) + [-v for v in ties.values()]
    assert list(deq) == want


def test_quantize_exhaustive_bf16_against_brute_force():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 7.96875)]
    w, nb = _block_with_scale_anchor(v)
    q, s = O.quantize(w)
    assert np.all(s == 127)
    codes = O.unpack_nibbles(q).reshape(nb, 32)[:, 1:].reshape(-1)[: len(v)]
    want = np.array([_brute_force_code(float(x)) for x in v], np.uint8)
    bad = np.nonzero(codes != want)[0]
    assert bad.size == 0, (v[bad[:5]], codes[bad[:5]], want[bad[:5]])


def test_quantize_scale_rule():
    rng = np.random.default_rng(1)
    amax = np.concatenate([2.0 ** rng.uniform(-60, 60, 4000), 2.0 ** np.arange(-40, 41)]).astype(np.float32)
    amax = amax[amax > 0]
    w = np.zeros((len(amax), 32), np.float32)
    w[:, 5] = -amax
    _, s = O.quantize(w)
    want = [min(254, max(0, math.floor(math.log2(float(a))) - 2 + 127)) for a in amax]
    assert list(s[:, 0]) == want
    # amax == 0 -> 127 and all-zero codes
    q0, s0 = O.quantize(np.zeros((1, 32), np.float32))
    assert s0[0, 0] == 127 and not q0.any()


def test_quantize_round_trip_of_representable_blocks():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, size=(64, 64)).astype(np.uint8)
    codes[:, 0] = rng.choice([6, 7, 14, 15], size=64)      # a magnitude 4 or 6 fixes the scale
    codes[:, 32] = rng.choice([6, 7, 14, 15], size=64)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = rng.integers(90, 160, size=(64, 2)).astype(np.uint8)
    w = O.dequant(q, s).astype(np.float32)
    q2, s2 = O.quantize(w)
    assert np.array_equal(s2, s)
    # -0.0 and +0.0 dequantise equal but keep their sign through fp32
    assert np.array_equal(O.dequant(q2, s2), O.dequant(q, s))


def test_quantize_idempotent_and_error_bound():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((32, 256)) * rng.uniform(1e-3, 10, size=(32, 1))).astype(np.float32)
    q, s = O.quantize(w)
    deq = O.dequant(q, s)
    q2, s2 = O.quantize(deq.astype(np.float32))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    X = np.repeat(O.e8m0_value(s), 32, axis=1)
    a = np.abs(w.astype(np.float64)) / X
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    err = np.abs(deq - w) / X
    ok = (err <= half_step) | (a > 6)
    assert ok.all()
    sat = a > 6
    assert np.all(np.abs(deq[sat]) == 6 * X[sat])


def test_quantize_keeps_sign_of_zero():
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 4.0
    w[0, 1] = -0.0
    w[0, 2] = -0.1          # rounds to -0
    q, _ = O.quantize(w)
    codes = O.unpack_nibbles(q)[0]
    assert codes[1] == 8 and codes[2] == 8 and codes[3] == 0


# ----------------------------------------------------------------------------- routing


def test_topk_matches_full_sort_and_gates():
    rng = np.random.default_rng(4)
    T, E, k = 16, 40, 6
    logits = rng.standard_normal((T, E))
    logits[3, 7] = logits[3, 2]          # an exact tie: lower index first
    idx, gate = O.topk_gates(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert list(idx[t]) == order
        z = logits[t, order]
        ref = scipy.special.softmax(z)
        assert np.allclose(gate[t], ref, rtol=0, atol=1e-15)
        assert abs(gate[t].sum() - 1) <= 1e-12
        assert np.all(np.diff(gate[t]) <= 0)


def test_topk_with_k_equal_E_is_full_softmax():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((3, 9))
    idx, gate = O.topk_gates(logits, 9)
    for t in range(3):
        full = scipy.special.softmax(logits[t])
        assert np.allclose(gate[t], full[idx[t]], atol=1e-15)


def test_assignment_invariants_and_brute_force():
    rng = np.random.default_rng(6)
    T, E, k = 12, 10, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = O.assignment(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert sorted(perm.tolist()) == list(range(T * k))
    pairs = sorted(((int(idx[t, j]), t, j) for t in range(T) for j in range(k)))
    assert perm.tolist() == [t * k + j for (_, t, j) in pairs]


# ----------------------------------------------------------------------------- experts


def _random_layer(rng, H, I, E, scale_lo=118, scale_hi=126):
    def mat(r, c):
        q = rng.integers(0, 256, size=(r, c // 2)).astype(np.uint8)
        s = rng.integers(scale_lo, scale_hi, size=(r, c // 32)).astype(np.uint8)
        return q, s
    return [dict(gate=mat(I, H), up=mat(I, H), down=mat(H, I)) for _ in range(E)]


def _mk(ex):
    return O.ExpertMatrices(*ex["gate"], *ex["up"], *ex["down"])


@pytest.mark.parametrize("T,H,I,E,k", [(8, 256, 128, 8, 2), (2, 128, 64, 6, 3)])
def test_sparse_equals_dense_masked_sum_over_all_experts(T, H, I, E, k):
    rng = np.random.default_rng(7)
    layer = _random_layer(rng, H, I, E)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) * 0.02
    b = rng.standard_normal(E) * 0.1
    out = O.moe_layer(x, wr, b, k, lambda e: _mk(layer[e]))
    # brute force: every expert on every token, masked by the routing
    logits = x @ wr.T + b
    dense = np.zeros_like(x)
    for e in range(E):
        m = _mk(layer[e])
        g_full = m.gate @ x.T           # [I, T]
        u_full = m.up @ x.T
        a = g_full * scipy.special.expit(g_full) * u_full
        d_full = (m.down @ a).T          # [T, H]
        for t in range(T):
            top = sorted(range(E), key=lambda j: (-logits[t, j], j))[:k]
            if e in top:
                gates = scipy.special.softmax(logits[t, top])
                dense[t] += gates[top.index(e)] * d_full[t]
    rel = np.linalg.norm(out["y"] - dense) / np.linalg.norm(dense)
    assert rel <= 1e-12


def test_top1_output_is_the_expert_ffn():
    rng = np.random.default_rng(8)
    H, I, E = 128, 64, 4
    layer = _random_layer(rng, H, I, E)
    x = rng.standard_normal((3, H))
    wr = rng.standard_normal((E, H))
    out = O.moe_layer(x, wr, None, 1, lambda e: _mk(layer[e]))
    for t in range(3):
        e = int(np.argmax(x[t] @ wr.T))
        assert out["gate"][t, 0] == 1.0
        assert np.array_equal(out["y"][t], _mk(layer[e]).ffn(x[t]))


def test_all_zero_nibbles_give_zero_output():
    rng = np.random.default_rng(9)
    H, I, E = 64, 32, 3
    layer = _random_layer(rng, H, I, E)
    for ex in layer:
        for name in ("gate", "up", "down"):
            ex[name] = (np.zeros_like(ex[name][0]), ex[name][1])
    out = O.moe_layer(rng.standard_normal((2, H)), rng.standard_normal((E, H)), None, 2, lambda e: _mk(layer[e]))
    assert not out["y"].any()


def test_constant_weights_closed_form():
    # every weight = +1.0 * 2^(s-127), x = c * ones:
    # gv = uv = H * c * 2^(sg-127); a = silu(gv) * uv; y_h = I * 2^(sd-127) * a (gates sum to 1)
    H, I, E, k, c = 64, 32, 3, 2, 0.375
    sg, sd = 120, 123
    ones = lambda r, cc, sb: (np.full((r, cc // 2), 0x22, np.uint8), np.full((r, cc // 32), sb, np.uint8))
    m = O.ExpertMatrices(*ones(I, H, sg), *ones(I, H, sg), *ones(H, I, sd))
    x = np.full((1, H), c)
    wr = np.random.default_rng(10).standard_normal((E, H))
    out = O.moe_layer(x, wr, None, k, lambda e: m)
    g = H * c * 2.0 ** (sg - 127)
    a = g / (1 + math.exp(-g)) * g
    want = I * 2.0 ** (sd - 127) * a
    assert np.allclose(out["y"], want, rtol=1e-14, atol=0)


def test_down_scale_plus_one_doubles_output_exactly():
    rng = np.random.default_rng(11)
    H, I, E, k = 128, 64, 5, 2
    layer = _random_layer(rng, H, I, E)
    x = rng.standard_normal((4, H))
    wr = rng.standard_normal((E, H))
    y1 = O.moe_layer(x, wr, None, k, lambda e: _mk(layer[e]))["y"]
    for ex in layer:
        q, s = ex["down"]
        ex["down"] = (q, (s + 1).astype(np.uint8))
    y2 = O.moe_layer(x, wr, None, k, lambda e: _mk(layer[e]))["y"]
    assert np.array_equal(y2, 2 * y1)


def test_silu_against_library_logistic():
    z = np.linspace(-30, 30, 601)
    assert np.allclose(O.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)


# ----------------------------------------------------------------------------- norm / stack


def test_rmsnorm_constant_row_and_library():
    H, c, eps = 64, -0.7, 1e-6
    w = np.linspace(0.5, 1.5, H)
    n = O.rmsnorm(np.full((1, H), c), w, eps)
    assert np.allclose(n[0], w * c / math.sqrt(c * c + eps), rtol=1e-15)
    rng = np.random.default_rng(12)
    r = rng.standard_normal((5, H))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(r), (H,), torch.from_numpy(w), eps=eps).numpy()
    assert np.allclose(O.rmsnorm(r, w, eps), ref, rtol=1e-14, atol=1e-15)


def test_stack_with_zero_experts_is_identity_and_residual_adds():
    rng = np.random.default_rng(13)
    H, I, E, k = 64, 32, 4, 2
    zero = _random_layer(rng, H, I, E)
    for ex in zero:
        ex["down"] = (np.zeros_like(ex["down"][0]), ex["down"][1])
    x = rng.standard_normal((3, H))
    L = [dict(wr=rng.standard_normal((E, H)), b=None, norm_w=np.ones(H), expert_fn=lambda e: _mk(zero[e]))] * 3
    assert np.array_equal(O.moe_stack(x, L, k, 1e-6)["y"], x)
    # one layer with live experts: r1 = x + MoE(norm(x))
    live = _random_layer(rng, H, I, E)
    wr = rng.standard_normal((E, H))
    w = rng.uniform(0.5, 1.5, H)
    L1 = [dict(wr=wr, b=None, norm_w=w, expert_fn=lambda e: _mk(live[e]))]
    got = O.moe_stack(x, L1, k, 1e-6)["y"]
    n = torch.nn.functional.rms_norm(torch.from_numpy(x), (H,), torch.from_numpy(w), eps=1e-6).numpy()
    want = x + O.moe_layer(n, wr, None, k, lambda e: _mk(live[e]))["y"]
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- metric


def test_bandwidth_bound_reproduces_page_numbers():
    for bw, wbytes, gpus, printed, dec in _golden_rows("bandwidth_bound.txt"):
        got = int(gpus) * O.implied_tokens_per_s(float(bw), float(wbytes))
        assert abs(got - float(printed)) <= 10.0 ** -int(dec), (bw, wbytes, gpus, got, printed)


def test_verify_tokens_per_s():
    # one verify forward per 6.30 accepted tokens: 1 ms per verify -> 6300 tokens/s
    assert O.verify_tokens_per_s(1e-3) == pytest.approx(6300.0)


# ----------------------------------------------------------------------------- verify acceptance


def _one_hot_logits(targets, V, base=0.0):
    """Logits whose greedy token at each position is the given one (value 1 vs base)."""
    S, B = targets.shape
    lg = np.full((S, B, V), base)
    for s in range(S):
        for i in range(B):
            lg[s, i, targets[s, i]] = 1.0
    return lg


def test_accept_block_hand_cases():
    # position i's logits predict the token of position i + 1 (DFlash verify, page 3)
    targets = np.array([[2, 3, 1, 4],     # drafts 2, 3 agree, draft 0 at position 3 does not
                        [1, 1, 2, 0],     # every draft agrees: 3 accepted + the target's token
                        [4, 0, 0, 0]])    # the first draft disagrees
    tokens = np.array([[9, 2, 3, 0],
                       [7, 1, 1, 2],
                       [5, 3, 0, 0]])
    r = O.accept_block(_one_hot_logits(targets, 5), tokens)
    assert r["target"].tolist() == targets.tolist()
    assert r["accepted"].tolist() == [3, 4, 1]       # tokens yielded per verify
    assert r["next_token"].tolist() == [1, 0, 4]     # the target's token after the accepted drafts


def test_accept_block_ties_nan_and_block_of_one():
    lg = np.zeros((1, 3, 6))
    lg[0, 0, [1, 4]] = 2.0               # tie: the lower token wins
    lg[0, 1, :] = [0.5, np.nan, 0.1, 0.7, -1.0, 0.7]   # NaN never wins; tie 3 / 5 -> 3
    lg[0, 2, 2] = 1.0
    r = O.accept_block(lg, np.array([[0, 1, 3]]))
    assert r["target"].tolist() == [[1, 3, 2]]
    assert r["accepted"].tolist() == [3] and r["next_token"].tolist() == [2]
    one = O.accept_block(np.zeros((2, 1, 4)), np.zeros((2, 1), dtype=np.int64))
    assert one["accepted"].tolist() == [1, 1] and one["next_token"].tolist() == [0, 0]
