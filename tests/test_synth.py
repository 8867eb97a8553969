"""Seeded input generator: determinism, shapes, distributions and the margin rule (CPU)."""
import numpy as np
import torch

from mxfp4_moe_expert_gb300.synth import WORKLOADS, derive_seed, expert_weight, make_inputs, splitmix64
from oracle import moe_oracle as O


def test_splitmix64_reference_values():
    # splitmix64 from state 0: the first outputs of the published generator
    # (state advanced by the golden gamma before each output)
    z, outs = 0, []
    for _ in range(3):
        outs.append(splitmix64(z))
        z = (z + 0x9E3779B97F4A7C15) & ((1 << 64) - 1)
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_distinct_streams():
    wl = WORKLOADS["tiny"]
    a, b = make_inputs(wl), make_inputs(wl)
    assert torch.equal(a.x, b.x) and torch.equal(a.layers[0].router_w, b.layers[0].router_w)
    assert derive_seed(1, "gate", 0, 0) != derive_seed(1, "up", 0, 0)
    w1 = expert_weight(wl, 0, 1, "gate")
    assert torch.equal(w1, expert_weight(wl, 0, 1, "gate"))
    assert not torch.equal(w1, expert_weight(wl, 0, 2, "gate"))


def test_shapes_and_distributions():
    wl = WORKLOADS["mid"]
    inp = make_inputs(wl)
    assert inp.x.shape == (wl.T, wl.H) and inp.x.dtype == torch.bfloat16
    L = inp.layers[0]
    assert L.router_w.shape == (wl.E, wl.H) and L.router_w.dtype == torch.bfloat16
    assert abs(float(L.router_w.float().std()) - 0.02) < 0.001
    w = expert_weight(wl, 0, 0, "down")
    assert w.shape == (wl.H, wl.I) and w.dtype == torch.float32
    assert abs(float(w.std()) * wl.I ** 0.5 - 1.0) < 0.01


def test_margin_rule_holds_on_every_token():
    for name in ("tiny", "large", "batched"):
        wl = WORKLOADS[name]
        inp = make_inputs(wl)
        x = O.bf16_to_f64(inp.x.view(torch.int16).numpy().view(np.uint16))
        wr = O.bf16_to_f64(inp.layers[0].router_w.view(torch.int16).numpy().view(np.uint16))
        z = O.router_logits(x, wr, inp.layers[0].router_b.double().numpy())
        assert min(O.topk_margin(z[t], wl.k) for t in range(wl.T)) >= wl.margin


def test_zipf_workload_is_skewed():
    wl = WORKLOADS["batched"]
    inp = make_inputs(wl)
    x = inp.x.double().numpy()
    wr = inp.layers[0].router_w.double().numpy()
    idx, _ = O.topk_gates(O.router_logits(x, wr, inp.layers[0].router_b.double().numpy()), wl.k)
    counts = np.bincount(idx.reshape(-1), minlength=wl.E)
    assert counts.max() >= 64          # a heavy head for the dense path
    assert (counts > 0).sum() >= 100   # and a long tail of cold experts
    assert ((counts > 0) & (counts <= 2)).sum() >= 40
