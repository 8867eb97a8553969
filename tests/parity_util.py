"""Helpers shared by the parity tests: oracle inputs from the seeded generator,
and the tolerance of the layer output.

Tolerance (stated by the workload definition): per token row, relative L2
error <= 5e-3 and max abs error <= 1e-2 * rms(reference row), against the fp64
oracle.  Routing indices and the token-expert grouping are compared bit-exact.
"""
from __future__ import annotations

import concurrent.futures
import json
import multiprocessing
import os

import numpy as np
import torch

from mxfp4_moe_expert_gb300.synth import Inputs, Workload, expert_weight
from oracle import moe_oracle as O

REL_L2 = 5e-3
MAX_ABS_RMS = 1e-2


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return O.bf16_to_f64(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def assert_rows_close(got: np.ndarray, ref: np.ndarray, rows=None, what=""):
    rows = range(ref.shape[0]) if rows is None else rows
    worst = (0.0, 0.0)
    for t in rows:
        r = ref[t]
        g = got[t]
        nrm = np.linalg.norm(r)
        rms = nrm / np.sqrt(r.size)
        rel = np.linalg.norm(g - r) / nrm if nrm > 0 else np.linalg.norm(g)
        mx = np.max(np.fabs(g - r)) / rms if rms > 0 else np.max(np.fabs(g))
        worst = (max(worst[0], rel), max(worst[1], mx))
        assert rel <= REL_L2, f"{what} row {t}: rel L2 {rel:.3e}"
        assert mx <= MAX_ABS_RMS, f"{what} row {t}: max abs / rms {mx:.3e}"
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "what": what,
                                "rows": len(rows), "worst_rel_l2": worst[0],
                                "worst_maxabs_over_rms": worst[1]}) + "\n")
    return worst


class OracleExperts:
    """Oracle-side experts of one layer: each routed expert's fp32 master weights
    are redrawn by the generator (on `weights_device`, the device the GPU side
    drew them on) and MXFP4-encoded by the oracle's own quantizer."""

    def __init__(self, wl: Workload, layer: int, weights_device="cpu", check_against=None):
        self.wl, self.layer, self.dev = wl, layer, weights_device
        self.check = check_against  # optional device layer dict: its bytes must equal the oracle's
        self.cache = {}

    def quantized(self, e: int):
        if e not in self.cache:
            out = {}
            for m in ("gate", "up", "down"):
                w = expert_weight(self.wl, self.layer, e, m, self.dev).cpu().numpy()
                q, s = O.quantize(w)
                if self.check is not None:
                    assert np.array_equal(self.check[m + "_q"][e].cpu().numpy(), q), (m, e)
                    assert np.array_equal(self.check[m + "_s"][e].cpu().numpy(), s), (m, e)
                out[m] = (q, s)
            self.cache[e] = out
        return self.cache[e]

    def __call__(self, e: int) -> O.ExpertMatrices:
        d = self.quantized(e)
        return O.ExpertMatrices(*d["gate"], *d["up"], *d["down"])


def oracle_quantizer_to(device):
    """Quantizer for device_layers that uses the oracle (CPU) and uploads the bytes."""
    def qz(w):
        q, s = O.quantize(w.cpu().numpy())
        return torch.from_numpy(q).to(device), torch.from_numpy(s).to(device)
    return qz


def oracle_layer_args(inputs: Inputs, layer: int):
    L = inputs.layers[layer]
    wr = bf16_np(L.router_w)
    b = L.router_b.double().numpy()
    nw = bf16_np(L.norm_w) if L.norm_w is not None else None
    return wr, b, nw


# ---- the oracle's encoding of many experts, in parallel -----------------------------


def _worker_init():
    torch.set_num_threads(1)


def _oracle_matrix_bytes(task):
    """Worker: one expert matrix drawn on the CPU and MXFP4-encoded by the oracle."""
    wl, layer, e, m = task
    q, s = O.quantize(expert_weight(wl, layer, e, m, "cpu").numpy())
    return layer, e, m, q, s


class OracleExpertBank:
    """The oracle's bytes of a workload's experts: fp32 master weights drawn by the
    generator on the CPU and encoded by oracle.quantize, one matrix per task in a pool of
    spawned processes (safe whether or not this process has touched the GPU); cached per
    (layer, expert).  The GPU side receives these same bytes (upload), so the library's
    quantizer plays no part in the comparison."""

    MATRICES = ("gate", "up", "down")

    def __init__(self, wl: Workload, workers: int | None = None):
        self.wl = wl
        self.cache = {}
        n = workers or max(1, min(48, os.cpu_count() or 1))
        self.pool = concurrent.futures.ProcessPoolExecutor(
            n, mp_context=multiprocessing.get_context("spawn"), initializer=_worker_init)

    def ensure(self, layer: int, experts) -> None:
        todo = sorted({int(e) for e in np.asarray(experts).reshape(-1)} - {e for (l, e) in self.cache if l == layer})
        tasks = [(self.wl, layer, e, m) for e in todo for m in self.MATRICES]
        got = {}
        for l, e, m, q, s in self.pool.map(_oracle_matrix_bytes, tasks, chunksize=1):
            got.setdefault(e, {})[m] = (q, s)
        for e, d in got.items():
            self.cache[(layer, e)] = d

    def expert_fn(self, layer: int):
        """expert_fn for the oracle's layer functions."""
        def fn(e):
            self.ensure(layer, [e])
            d = self.cache[(layer, int(e))]
            return O.ExpertMatrices(*d["gate"], *d["up"], *d["down"])
        return fn

    def upload(self, layer_tensors: dict, layer: int) -> int:
        """Writes every cached expert of `layer` into a device layer (dict of [E, ...]
        tensors); returns how many experts were written."""
        n = 0
        for (l, e), d in self.cache.items():
            if l != layer:
                continue
            for m in self.MATRICES:
                q, s = d[m]
                layer_tensors[m + "_q"][e].copy_(torch.from_numpy(q))
                layer_tensors[m + "_s"][e].copy_(torch.from_numpy(s))
            n += 1
        return n

    def close(self):
        self.pool.shutdown(cancel_futures=True)
