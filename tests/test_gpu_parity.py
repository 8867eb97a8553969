"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Routing indices and the token-expert grouping must be bit-exact; each output
row must meet rel L2 <= 5e-3 and max abs <= 1e-2 * rms(ref row).  Inputs are
the seeded workloads; the oracle always encodes weights with its own
quantizer (the device copy may come from the library's quantizer only after
its bytes are shown equal to the oracle's).
"""
import numpy as np
import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from mxfp4_moe_expert_gb300.synth import WORKLOADS, Workload, expert_weight, make_inputs
from mxfp4_moe_expert_gb300.workload import device_layers, repack
from oracle import moe_oracle as O
from parity_util import (OracleExpertBank, OracleExperts, assert_rows_close, bf16_np, oracle_layer_args,
                         oracle_quantizer_to)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()


def _moe(wl, layers, flags=0, **kw):
    if wl.norm:
        flags |= pkg.MOE_FLAG_NORM
    return pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T,
                         layers=layers, flags=flags, rms_eps=wl.rms_eps, **kw)


def _run(moe, x, T=None):
    T = x.shape[0] if T is None else T
    bufs, dbg = moe.debug_buffers(T)
    y = moe.forward(x, dbg=dbg, check=True)
    torch.cuda.synchronize()
    return y, {k: v.cpu().numpy() for k, v in bufs.items()}


def _check_routing(dbgl, ref, what="", deep=False):
    """Indices and grouping bit-exact.  Gates: a layer that sees the exact input
    (the first) within fp32 rounding of the softmax; a deeper layer of a stack
    sees a residual that already carries the earlier layers' output error (each
    within the stated output tolerance), which moves its logits by ~1e-4 and its
    gates by ~1e-5 .. 1e-4, so they are compared within 5e-4."""
    assert np.array_equal(dbgl["idx"], ref["idx"]), what
    assert np.array_equal(dbgl["counts"], ref["counts"]), what
    assert np.array_equal(dbgl["offsets"], ref["offsets"]), what
    assert np.array_equal(dbgl["perm"], ref["perm"]), what
    if deep:
        assert np.allclose(dbgl["gate"], ref["gate"], rtol=0, atol=5e-4), what
    else:
        assert np.allclose(dbgl["gate"], ref["gate"], rtol=1e-5, atol=1e-6), what


def _dbg_layer(bufs, l):
    return dict(idx=bufs["topk_idx"][l], gate=bufs["topk_gate"][l], counts=bufs["expert_counts"][l],
                offsets=bufs["expert_offsets"][l], perm=bufs["perm"][l])


# ----------------------------------------------------------------------------- quantizer


def test_quantize_kernel_bit_exact():
    g = torch.Generator().manual_seed(11)
    w = torch.randn((96, 1024), generator=g) * torch.exp2(torch.randint(-30, 30, (96, 1), generator=g).float())
    w[0, :32] = 0.0
    w[1, :32] = -0.0
    w[2, :32] = torch.tensor([4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4) * torch.tensor([1.0, -1.0] * 16)
    w[3, :32] = 1e-42                         # subnormal block
    w[4, :32] = 3.0e38                        # near the fp32 maximum
    w[5, 0] = 7.99
    q_ref, s_ref = O.quantize(w.numpy())
    q, s = pkg.quantize(w.to(DEV))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantize_kernel_matches_oracle_on_expert_weights():
    wl = WORKLOADS["mid"]
    w = expert_weight(wl, 0, 5, "down", DEV)
    q, s = pkg.quantize(w)
    q_ref, s_ref = O.quantize(w.cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(s.cpu().numpy(), s_ref)


# ----------------------------------------------------------------------------- full oracle, small shapes


# Shapes whose H and I are multiples of 512 run the TMA expert kernel; the others
# run the multi-kernel path.
SMALL = [
    WORKLOADS["tiny"],
    Workload("ragged", T=13, H=1024, I=384, E=16, k=4, seed=0x5EED0100),
    Workload("top1", T=5, H=512, I=256, E=6, k=1, seed=0x5EED0101),
    Workload("k_eq_E", T=3, H=256, I=128, E=4, k=4, seed=0x5EED0102),
    Workload("one_token", T=1, H=768, I=512, E=32, k=8, seed=0x5EED0103),
    Workload("tma_ragged", T=13, H=1024, I=512, E=16, k=4, seed=0x5EED0110),
    Workload("tma_top1", T=5, H=512, I=512, E=6, k=1, seed=0x5EED0111),
    Workload("tma_k_eq_E", T=3, H=512, I=1024, E=4, k=4, seed=0x5EED0112),
    Workload("tma_one_token", T=1, H=1536, I=512, E=32, k=8, seed=0x5EED0113),
    Workload("tma_many_tokens", T=40, H=512, I=512, E=4, k=2, seed=0x5EED0114),
    # 64 pairs over 4 experts: several 8-pair chunks per expert in the shared-memory routing path
    Workload("tma_multi_chunk", T=32, H=512, I=512, E=4, k=2, seed=0x5EED0116),
    # the largest block of the persistent path: T * k = 4096 pairs (512 chunks), routed through
    # the workspace, every router token block and the combine's shared-memory pair table full
    Workload("tma_max_pairs", T=512, H=512, I=512, E=16, k=8, seed=0x5EED0118),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_layer_parity_full_oracle(wl):
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe = _moe(wl, layers)
    y, bufs = _run(moe, inputs.x.to(DEV))
    wr, b, _ = oracle_layer_args(inputs, 0)
    ref = O.moe_layer(bf16_np(inputs.x), wr, b, wl.k, OracleExperts(wl, 0, "cpu"))
    _check_routing(_dbg_layer(bufs, 0), ref, wl.name)
    assert_rows_close(y.double().cpu().numpy(), ref["y"], what=wl.name)
    moe.close()


@pytest.mark.parametrize("wl", [w for w in SMALL if w.H % 512 == 0 and w.I % 512 == 0], ids=lambda w: w.name)
def test_layer_parity_packed_experts(wl):
    """The same layers with the experts read from the packed copy only (the canonical
    tensors are dropped from the layer): persistent forward and one-launch-per-phase
    forward, against the oracle on every row."""
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV),
                                   packed=True)
    for m in ("gate", "up", "down"):
        layers[0][m + "_q"] = layers[0][m + "_s"] = None
    wr, b, _ = oracle_layer_args(inputs, 0)
    ref = O.moe_layer(bf16_np(inputs.x), wr, b, wl.k, OracleExperts(wl, 0, "cpu"))
    for flags in (0, pkg.MOE_FLAG_MULTI_KERNEL):
        moe = _moe(wl, layers, flags=flags)
        y, bufs = _run(moe, inputs.x.to(DEV))
        _check_routing(_dbg_layer(bufs, 0), ref, f"{wl.name} packed flags={flags}")
        assert_rows_close(y.double().cpu().numpy(), ref["y"], what=f"{wl.name} packed flags={flags}")
        moe.close()


@pytest.mark.parametrize("wl", [w for w in SMALL if w.name in ("tma_many_tokens", "tma_max_pairs")], ids=lambda w: w.name)
def test_gathered_blocks_with_and_without_the_dense_operand(wl):
    """Blocks routed through the workspace run chunks of 32 pairs x 4 E2M1 terms (dense
    operand) by default and of 16 pairs x 8 terms with MOE_FLAG_NO_DENSE: both against the
    oracle on every row, and the 8-term result nearer to it."""
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV),
                                   packed=True)
    wr, b, _ = oracle_layer_args(inputs, 0)
    ref = O.moe_layer(bf16_np(inputs.x), wr, b, wl.k, OracleExperts(wl, 0, "cpu"))
    worst = {}
    for flags in (0, pkg.MOE_FLAG_NO_DENSE):
        moe = _moe(wl, layers, flags=flags)
        y, bufs = _run(moe, inputs.x.to(DEV))
        _check_routing(_dbg_layer(bufs, 0), ref, f"{wl.name} flags={flags}")
        worst[flags] = assert_rows_close(y.double().cpu().numpy(), ref["y"], what=f"{wl.name} flags={flags}")
        moe.close()
    assert worst[pkg.MOE_FLAG_NO_DENSE][0] < worst[0][0]


@pytest.mark.parametrize("wl", [
    Workload("stack_small", T=6, H=512, I=256, E=12, k=3, layers=4, norm=True, seed=0x5EED0104),
    Workload("stack_tma", T=7, H=1024, I=512, E=12, k=3, layers=3, norm=True, seed=0x5EED0115),
    # 96 pairs: routed through the workspace, input operand gathered per chunk, residual stack
    Workload("stack_tma_large_block", T=24, H=1024, I=512, E=12, k=4, layers=2, norm=True, seed=0x5EED0117),
], ids=lambda w: w.name)
def test_stack_parity_small(wl):
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe = _moe(wl, layers)
    y, bufs = _run(moe, inputs.x.to(DEV))
    L = []
    for l in range(wl.layers):
        wr, b, nw = oracle_layer_args(inputs, l)
        L.append(dict(wr=wr, b=b, norm_w=nw, expert_fn=OracleExperts(wl, l, "cpu")))
    ref = O.moe_stack(bf16_np(inputs.x), L, wl.k, wl.rms_eps)
    for l in range(wl.layers):
        margins = [O.topk_margin(ref["layers"][l]["logits"][t], wl.k) for t in range(wl.T)]
        assert min(margins) > 1e-5, (l, min(margins))
        _check_routing(_dbg_layer(bufs, l), ref["layers"][l], f"layer {l}", deep=l > 0)
    assert_rows_close(y.double().cpu().numpy(), ref["y"], what="stack")
    moe.close()


def test_wide_dynamic_range_activations():
    """Every element of x carries an extra factor 2^u, u uniform in [-20, 20], so one
    32-element MX block of x spans up to 2^40 in magnitude: the worst case of the
    expert operand's 8-term E2M1 split, whose terms represent each value relative to
    its block's maximum (values far below the block maximum are dropped).  The layer
    output must still meet the output tolerance on every row.  The router logits reach
    ~1e5 here, where fp32 accumulation moves them by up to ~1, so the margin condition
    on the input is 16 instead of 1e-3."""
    wl = Workload("wide_x", T=13, H=1024, I=512, E=16, k=4, seed=0x5EED0119, x_spread=20, margin=16.0)
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    xf = bf16_np(inputs.x)
    blocks = np.abs(xf).reshape(wl.T, -1, 32)
    nz = np.where(blocks > 0, blocks, np.nan)
    assert np.nanmax(np.log2(np.nanmax(nz, axis=2) / np.nanmin(nz, axis=2))) >= 30   # the spread is really there
    moe = _moe(wl, layers)
    y, bufs = _run(moe, inputs.x.to(DEV))
    wr, b, _ = oracle_layer_args(inputs, 0)
    with np.errstate(over="ignore"):   # silu of very negative gate values: exp overflows to inf, silu -> -0
        ref = O.moe_layer(xf, wr, b, wl.k, OracleExperts(wl, 0, "cpu"))
    _check_routing(_dbg_layer(bufs, 0), ref, wl.name)
    assert_rows_close(y.double().cpu().numpy(), ref["y"], what=wl.name)
    moe.close()


def test_cuda_graph_replay_of_per_phase_forward():
    """The one-launch-per-phase forward (the comparison path for per-operator execution)
    captured once in a CUDA graph and replayed: each replay's output matches the fp64
    oracle, and equals the eagerly launched forward bit for bit."""
    wl = SMALL[5]
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe = _moe(wl, layers, flags=pkg.MOE_FLAG_MULTI_KERNEL)
    x = inputs.x.to(DEV)
    eager = moe.forward(x, check=True)
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device=DEV)
    ws = moe.new_workspace(wl.T)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.forward(x, y, ws, side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        moe.forward(x, y, ws, side.cuda_stream)
    torch.cuda.synchronize()
    wr, b, _ = oracle_layer_args(inputs, 0)
    ref = O.moe_layer(bf16_np(inputs.x), wr, b, wl.k, OracleExperts(wl, 0, "cpu"))
    for replay in range(2):
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkg.moe_mxfp4_check(moe.handle, ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == pkg.MOE_OK
        assert torch.equal(y, eager), replay
        assert_rows_close(y.double().cpu().numpy(), ref["y"], what=f"graph replay {replay}")
    del graph
    moe.close()


def test_bf16_output_and_host_entry_point():
    wl = SMALL[1]
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe32 = _moe(wl, layers)
    y32 = moe32.forward(inputs.x.to(DEV), check=True)
    moe16 = _moe(wl, layers, flags=pkg.MOE_FLAG_OUT_BF16)
    y16 = moe16.forward(inputs.x.to(DEV), check=True)
    assert y16.dtype == torch.bfloat16
    assert torch.equal(y16, y32.to(torch.bfloat16))
    ws = moe32.new_workspace(wl.T)
    xh = inputs.x.clone().pin_memory()
    yh = torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory()
    moe32.forward_host(xh, yh, ws)
    assert torch.equal(yh, y32.cpu())
    moe32.close()
    moe16.close()


@pytest.mark.parametrize("wl", [SMALL[0], SMALL[5]], ids=lambda w: w.name)
def test_tma_and_multi_kernel_paths_agree(wl):
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    x = inputs.x.to(DEV)
    a = _moe(wl, layers).forward(x, check=True)
    b = _moe(wl, layers, flags=pkg.MOE_FLAG_MULTI_KERNEL).forward(x, check=True)
    assert_rows_close(a.double().cpu().numpy(), b.double().cpu().numpy(), what="paths")


@pytest.mark.parametrize("wl", [SMALL[1], SMALL[5]], ids=lambda w: w.name)
def test_expert_shards_sum_to_full_layer(wl):
    """Expert-parallel shards (disjoint expert ranges) sum to the full layer; in the
    persistent forward (SMALL[5]) some tokens have no slot in a shard, whose output rows
    no down item writes."""
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    x = inputs.x.to(DEV)
    full = _moe(wl, layers).forward(x, check=True)
    parts = [_moe(wl, layers, expert_begin=b, expert_end=e).forward(x, check=True) for b, e in ((0, 5), (5, 11), (11, 16))]
    total = parts[0].double() + parts[1].double() + parts[2].double()
    assert_rows_close(total.cpu().numpy(), full.double().cpu().numpy(), what="shards")


@pytest.mark.parametrize("wl", [SMALL[0], SMALL[5]], ids=lambda w: w.name)
def test_down_scale_plus_one_doubles_output_exactly(wl):
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    x = inputs.x.to(DEV)
    y1 = _moe(wl, layers).forward(x, check=True)
    L2 = dict(layers[0])
    L2["down_s"] = layers[0]["down_s"] + 1
    y2 = _moe(wl, [L2]).forward(x, check=True)
    assert torch.equal(y2, 2 * y1)


@pytest.mark.parametrize("wl", [SMALL[0], SMALL[5]], ids=lambda w: w.name)
def test_nan_scale_of_a_routed_expert_is_reported(wl):
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe = _moe(wl, layers)
    bufs, dbg = moe.debug_buffers(wl.T)
    moe.forward(inputs.x.to(DEV), dbg=dbg, check=True)
    e = int(bufs["topk_idx"][0, 0, 0])
    L2 = dict(layers[0])
    L2["up_s"] = layers[0]["up_s"].clone()
    L2["up_s"][e, 3, 1] = 0xFF
    bad = _moe(wl, [L2])
    with pytest.raises(pkg.MoeError) as ei:
        bad.forward(inputs.x.to(DEV), check=True)
    assert ei.value.status == pkg.MOE_ERR_BAD_SCALE


def test_empty_and_invalid_calls():
    wl = SMALL[0]
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    moe = _moe(wl, layers)
    ws = moe.new_workspace(wl.T)
    st = torch.cuda.current_stream().cuda_stream
    x = inputs.x.to(DEV)
    y = torch.zeros((wl.T, wl.H), device=DEV)
    assert pkg.moe_mxfp4_forward(moe.handle, x.data_ptr(), 0, y.data_ptr(), ws.data_ptr(), ws.numel(), st) == 0
    assert pkg.moe_mxfp4_forward(moe.handle, x.data_ptr(), wl.T + 1, y.data_ptr(), ws.data_ptr(), ws.numel(),
                                 st) == pkg.MOE_ERR_INVALID_ARG
    assert pkg.moe_mxfp4_forward(moe.handle, x.data_ptr(), wl.T, y.data_ptr(), ws.data_ptr(), ws.numel() - 256,
                                 st) == pkg.MOE_ERR_WORKSPACE
    assert pkg.moe_mxfp4_forward(moe.handle, x.data_ptr(), wl.T, y.data_ptr(), ws.data_ptr() + 16, ws.numel() - 256,
                                 st) == pkg.MOE_ERR_WORKSPACE
    L2 = dict(layers[0])
    L2["gate_q"] = torch.empty(wl.E * wl.I * wl.H // 2 + 16, dtype=torch.uint8, device=DEV)[8:]
    with pytest.raises(pkg.MoeError):
        _moe(wl, [L2])
    moe.close()


# ----------------------------------------------------------------------------- full sizes
#
# Oracle first: the routing of the block comes from the oracle; the experts that the
# checked rows route to are drawn on the CPU and encoded by the oracle's quantizer (in
# parallel, OracleExpertBank), and exactly those bytes are written into the device layer
# (whose other experts hold GPU-drawn weights encoded by the library's quantizer: no
# checked row reads them, and a mis-routed pair would fail the bit-exact routing check
# first).  The device forward then runs the whole block in the launch configuration the
# benchmark times.


def _layer_full_size(name, rows=None, packed=True):
    """Single layer at full size: routing of every token bit-exact (indices, counts,
    offsets, perm; gates within 1e-5), and every row in `rows` (default: all) within the
    output tolerance of the fp64 oracle.  packed: the experts are streamed from the
    packed copy (the layout the benchmark times)."""
    wl = WORKLOADS[name]
    inputs = make_inputs(wl)
    xf = bf16_np(inputs.x)
    wr, b, _ = oracle_layer_args(inputs, 0)
    idx, gate = O.topk_gates(O.router_logits(xf, wr, b), wl.k)
    counts, offsets, perm = O.assignment(idx, wl.E)
    rows = list(range(wl.T)) if rows is None else sorted(set(int(t) for t in rows))
    bank = OracleExpertBank(wl)
    try:
        bank.ensure(0, idx[rows])
        _, layers = device_layers(wl, inputs=inputs, device=DEV)
        assert bank.upload(layers[0], 0) == len(np.unique(idx[rows]))
        if packed:
            repack(layers, wl)
        moe = _moe(wl, layers)
        y, bufs = _run(moe, inputs.x.to(DEV))
        _check_routing(_dbg_layer(bufs, 0), dict(idx=idx, gate=gate, counts=counts, offsets=offsets, perm=perm), name)
        ref = O.moe_layer(xf[rows], wr, b, wl.k, bank.expert_fn(0))
        assert np.array_equal(ref["idx"], idx[rows])
        assert_rows_close(y.double().cpu().numpy()[rows], ref["y"], what=f"{name} ({len(rows)} rows)")
        moe.close()
        del layers
    finally:
        bank.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("packed", [True, False], ids=["packed", "canonical"])
def test_mid_layer_all_rows(packed):
    _layer_full_size("mid", packed=packed)


def test_large_layer_all_rows():
    _layer_full_size("large")


DENSE_CHUNK = 32   # pairs per chunk of a block routed through the workspace (4 E2M1 terms each)


def batched_rows(wl, idx, n_hot=3, n_total=48, seed=7):
    """Rows of the 256-token Zipf block to compare: every token of the first and of the
    last chunk (DENSE_CHUNK pairs, the chunking the kernel uses) of the most popular expert,
    the first and last 8 pairs of the next n_hot - 1 experts (the chunks that reuse those
    experts' weight rows most), tokens 0 and T-1, then seeded random tokens up to n_total."""
    counts, offsets, perm = O.assignment(idx, wl.E)
    rows = {0, wl.T - 1}
    for rank, e in enumerate(np.argsort(-counts, kind="stable")[:n_hot]):
        pairs = perm[offsets[e]:offsets[e + 1]]
        if rank == 0:
            last = (len(pairs) - 1) // DENSE_CHUNK * DENSE_CHUNK
            ends = (pairs[:DENSE_CHUNK], pairs[last:])
        else:
            ends = (pairs[:8], pairs[-8:])
        for chunk in ends:
            rows.update(int(p) // wl.k for p in chunk)
    rng = np.random.default_rng(seed)
    for t in rng.permutation(wl.T):
        if len(rows) >= n_total:
            break
        rows.add(int(t))
    return sorted(rows)


def test_batched_layer_rows():
    wl = WORKLOADS["batched"]
    inputs = make_inputs(wl)
    wr, b, _ = oracle_layer_args(inputs, 0)
    idx, _ = O.topk_gates(O.router_logits(bf16_np(inputs.x), wr, b), wl.k)
    rows = batched_rows(wl, idx)
    assert len(rows) >= 32
    _layer_full_size("batched", rows)


def stack_inputs_all_layers_conditioned(wl, bank):
    """The stack's input with every layer's top-(k+1) logit gaps >= wl.margin along the
    oracle trajectory of every token: a row of x is re-drawn (seeded) until the fp64
    trajectory of that token through all layers keeps the margin in each layer.  The
    layer is per token, so each row is decided on its own trajectory."""
    base = make_inputs(wl)   # router and norm weights do not depend on the rows of x
    args = [oracle_layer_args(base, l) for l in range(wl.layers)]
    for l in range(wl.layers):   # every expert of every layer: the trajectories may route anywhere
        bank.ensure(l, range(wl.E))

    def accept(t, row):
        r = bf16_np(row)[None]
        for l, (wr, b, nw) in enumerate(args):
            n = O.rmsnorm(r, nw, wl.rms_eps)
            if O.topk_margin(O.router_logits(n, wr, b)[0], wl.k) < wl.margin:
                return False
            r = r + O.moe_layer(n, wr, b, wl.k, bank.expert_fn(l))["y"]
        return True

    return make_inputs(wl, accept_row=accept), args


def test_stack_all_tokens_all_layers():
    """8 layers x 8 tokens at full size: the input conditioned on every layer's margin,
    then every layer's routing bit-exact for every token and every output row within
    the tolerance of the fp64 oracle's stack."""
    wl = WORKLOADS["stack"]
    bank = OracleExpertBank(wl)
    try:
        inputs, args = stack_inputs_all_layers_conditioned(wl, bank)
        xf = bf16_np(inputs.x)
        L = [dict(wr=wr, b=b, norm_w=nw, expert_fn=bank.expert_fn(l)) for l, (wr, b, nw) in enumerate(args)]
        ref = O.moe_stack(xf, L, wl.k, wl.rms_eps)
        for l in range(wl.layers):
            m = min(O.topk_margin(ref["layers"][l]["logits"][t], wl.k) for t in range(wl.T))
            assert m >= wl.margin, (l, m)
        _, layers = device_layers(wl, inputs=inputs, device=DEV)
        for l in range(wl.layers):
            bank.upload(layers[l], l)
        repack(layers, wl)
        moe = _moe(wl, layers)
        y, bufs = _run(moe, inputs.x.to(DEV))
        for l in range(wl.layers):
            _check_routing(_dbg_layer(bufs, l), ref["layers"][l], f"stack layer {l}", deep=l > 0)
        assert_rows_close(y.double().cpu().numpy(), ref["y"], what="stack (8 layers, all rows)")
        moe.close()
        del layers
    finally:
        bank.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("flags", [0, pkg.MOE_FLAG_MULTI_KERNEL], ids=["persistent", "multi_kernel"])
def test_device_wait_timeout_is_reported_and_context_survives(flags):
    """MOE_FLAG_DEBUG_STALL withholds one device-side signal (a grid-barrier arrival,
    or the completion of one expert's gate/up items), so the waits that depend on it
    run out after timeout_us (20 ms here): the kernel leaves and the status word says
    MOE_ERR_TIMEOUT.  The next forward on the same device then runs normally."""
    wl = SMALL[5]
    inputs, layers = device_layers(wl, device=DEV, weights_device="cpu", quantizer=oracle_quantizer_to(DEV))
    x = inputs.x.to(DEV)
    ref = _moe(wl, layers, flags=flags).forward(x, check=True)
    stalled = _moe(wl, layers, flags=flags | pkg.MOE_FLAG_DEBUG_STALL, timeout_us=20000)
    with pytest.raises(pkg.MoeError) as ei:
        stalled.forward(x, check=True)
    assert ei.value.status == pkg.MOE_ERR_TIMEOUT
    again = _moe(wl, layers, flags=flags).forward(x, check=True)
    assert torch.equal(again, ref)
