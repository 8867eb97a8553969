"""Benchmark of one MoE layer over an 8-token verify block (MXFP4 experts).

`python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large] [--impl reference]`

A step is one forward of the whole layer (routing, grouping, expert FFN,
combine) on seeded synthetic inputs resident in HBM.  The metric is
microseconds per MoE layer per verify block (lower is better), reported with
the achieved HBM bandwidth over the layer's algorithmic bytes (the routed
experts' nibbles and scales, router weights, x read, y written) and its
fraction of the measured copy bandwidth.  By default L2 is not flushed between
timed steps: every step's inputs (the routed experts' weights, 1.4 GB on the
384-expert layer) are over ten times larger than L2, so they stream from HBM each
step, while the kernel's code stays cached as it does in a decode loop; with
`--flush clean` a 256 MiB write and a 256 MiB read before each step (outside the
per-step events) also evict the code and every buffer.  Prints one JSON line.

The line also carries the same K steps timed under the other L2 protocol
(`l2_other_protocol`: not flushed when the main value is flushed, and the
reverse), the fractions of the measured copy bandwidth and of the nominal ~8 TB/s
HBM3e bandwidth, and `cpu_baseline`: the fp64 oracle timed over the whole verify
block (every routed expert) on all host cores.

`--impl reference` times that oracle harness (OracleHost) over K steps and prints
the same kind of line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# the CPU oracle legs run one worker process per host core, each single-threaded (BLAS included)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ACCEPTANCE_LENGTH = 6.30   # coding-task average accepted tokens per verify (page 3, "DFlash")
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e nominal bandwidth (~8 TB/s), the roofline the target is stated against


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str = ""):
        self.index = index
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _oracle_worker(conn, wl, experts_per_layer):
    """Worker process of OracleHost: encodes its experts once with the oracle's quantizer,
    then evaluates the oracle's expert FFN for the (pair, input row) lists it is sent."""
    import torch

    from mxfp4_moe_expert_gb300.synth import expert_weight
    from oracle import moe_oracle as O

    torch.set_num_threads(1)
    enc = {(l, e): [a for m in ("gate", "up", "down") for a in O.quantize(expert_weight(wl, l, e, m).numpy())]
           for l, es in enumerate(experts_per_layer) for e in es}
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        out = {}
        for (l, e), items in msg.items():
            m = O.ExpertMatrices(*enc[(l, e)])   # the oracle dequantises per forward, as in moe_layer
            for pid, xrow in items:
                out[pid] = m.ffn(xrow)
        conn.send(out)


class OracleHost:
    """The fp64 oracle's forward of a verify block on the host cores.  Routing (router
    logits, top-k, grouping), RMSNorm and the gate-weighted combine run in this process
    with the oracle's functions; the routed experts' SwiGLU FFNs (the oracle's
    ExpertMatrices) run in `workers` spawned processes, each owning a fixed share of the
    block's routed experts, encoded once before timing.  Every routed expert of the block
    is evaluated (no sampling)."""

    def __init__(self, wl, workers=None):
        import multiprocessing as mp

        import numpy as np
        import torch

        from mxfp4_moe_expert_gb300.synth import make_inputs
        from oracle import moe_oracle as O

        self.O, self.np, self.wl = O, np, wl
        inputs = make_inputs(wl)
        b16 = lambda t: O.bf16_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))
        self.x = b16(inputs.x)
        self.layers = [(b16(L.router_w), L.router_b.double().numpy(), b16(L.norm_w) if L.norm_w is not None else None)
                       for L in inputs.layers]
        # the routed experts of every layer along the oracle's own trajectory (outside the timing)
        routed = self._trajectory_experts()
        self.n = workers or max(1, os.cpu_count() or 1)
        self.owner = {}
        shares = [[[] for _ in range(wl.layers)] for _ in range(self.n)]
        i = 0
        for l, es in enumerate(routed):
            for e in es:
                shares[i % self.n][l].append(e)
                self.owner[(l, e)] = i % self.n
                i += 1
        self.owned = sum(len(es) for es in routed)
        self.routed = [0] * wl.layers   # routed experts per layer of the last forward
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for w in range(self.n):
            a_, b_ = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(b_, wl, shares[w]), daemon=True)
            pr.start()
            self.conns.append(a_)
            self.procs.append(pr)
        for c in self.conns:
            assert c.recv() == "ready"

    def _trajectory_experts(self):
        """Experts the workers own, per layer: a single layer's routed experts (its routing
        needs only the router); every expert of every layer of a stack (its later layers
        route a residual that depends on the expert outputs)."""
        O, wl = self.O, self.wl
        if wl.layers == 1:
            idx, _ = O.topk_gates(O.router_logits(self.x, *self.layers[0][:2]), wl.k)
            return [sorted(set(int(e) for e in idx.reshape(-1)))]
        return [list(range(wl.E)) for _ in range(wl.layers)]

    def forward(self):
        """One timed forward of the block; returns y (fp64 [T, H])."""
        O, np, wl = self.O, self.np, self.wl
        r = self.x.copy()
        for l, (wr, b, nw) in enumerate(self.layers):
            xin = O.rmsnorm(r, nw, wl.rms_eps) if wl.norm else r
            idx, gate = O.topk_gates(O.router_logits(xin, wr, b), wl.k)
            counts, offsets, perm = O.assignment(idx, wl.E)
            msgs = [dict() for _ in range(self.n)]
            self.routed[l] = int((counts > 0).sum())
            for e in np.nonzero(counts)[0]:
                items = [(int(p), xin[int(p) // wl.k]) for p in perm[offsets[e]:offsets[e + 1]]]
                msgs[self.owner[(l, int(e))]][(l, int(e))] = items
            for c, m in zip(self.conns, msgs):
                c.send(m)
            d = {}
            for c in self.conns:
                d.update(c.recv())
            y = np.zeros_like(xin)
            for t in range(wl.T):
                for j in range(wl.k):   # slot order, as the oracle's moe_layer
                    y[t] += gate[t, j] * d[t * wl.k + j]
            r = r + y if wl.norm else y
        return r

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except Exception:
                pass
        for pr in self.procs:
            pr.join(timeout=10)


def run_reference(args):
    """The oracle, as it stands, on the host cores (OracleHost): every routed expert of
    one verify block per step."""
    ws, rank = _dist()
    if rank != 0:
        return
    from mxfp4_moe_expert_gb300.synth import WORKLOADS

    wl = WORKLOADS[args.workload]
    host = OracleHost(wl)
    try:
        for _ in range(args.warmup):
            host.forward()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            host.forward()
            times.append(time.perf_counter() - t0)
    finally:
        host.close()
    us = statistics.mean(times) * 1e6 / wl.layers
    sample = (f"the whole {wl.T}-token verify block: all {sum(host.routed)} routed experts "
              f"({wl.layers} layer{'s' if wl.layers > 1 else ''}), no sampling; {host.n} worker processes")
    line = {
        "impl": "reference", "metric": "us_per_moe_layer_per_verify_block", "value": round(us, 1), "unit": "us",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us * wl.layers / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "layers": wl.layers},
        "cpu_baseline": {"value": round(us, 1), "unit": "us", "cores": host.n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_gpu(args):
    import numpy as np
    import torch

    import mxfp4_moe_expert_gb300 as pkg
    from mxfp4_moe_expert_gb300.synth import WORKLOADS
    from mxfp4_moe_expert_gb300.workload import device_layers, touched_bytes

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()

    wl = WORKLOADS[args.workload]
    if args.experts:
        wl = wl.scaled(E=args.experts, name=f"{wl.name}_E{args.experts}")
    packed = args.layout == "packed" and moe_tma(wl)
    inputs, layers = device_layers(wl, device=dev, packed=packed)   # the one-time repack is outside the timed region
    flags = pkg.MOE_FLAG_NORM if wl.norm else 0
    persistent = args.path == "persistent" and moe_tma(wl)
    if args.path in ("multi", "graph"):
        flags |= pkg.MOE_FLAG_MULTI_KERNEL
    moe = pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T, layers=layers,
                        flags=flags, rms_eps=wl.rms_eps)
    x = inputs.x.to(dev)
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device=dev)
    wsp = moe.new_workspace(wl.T, dev)
    stream = torch.cuda.current_stream(dev)
    st = stream.cuda_stream

    # routing of this input: the algorithmic bytes of one step
    bufs, dbg = moe.debug_buffers(wl.T, dev)
    moe.forward(x, y, wsp, st, dbg, check=True)
    counts = bufs["expert_counts"].cpu()
    alg_bytes = touched_bytes(wl, [counts[l] for l in range(wl.layers)])
    n_active = [int((counts[l] > 0).sum()) for l in range(wl.layers)]

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    graph = None
    if args.path == "graph":
        # the one-launch-per-phase forward captured once and replayed: the launch gaps of
        # the per-operator model without the persistent kernel
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                moe.forward(x, y, wsp, side.cuda_stream)
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            moe.forward(x, y, wsp, side.cuda_stream)
        torch.cuda.synchronize()

    def flush_l2(i, mode=args.flush):
        # "write": a 256 MiB write (L2 is 129 MB) leaves L2 full of dirty lines of the
        # flush buffer; "clean" then reads another 256 MiB buffer, so the write-back of
        # those lines happens here and the timed forward starts from a clean, cold L2
        if mode == "none":
            return
        flush.fill_(i & 0xFF)
        if mode == "clean":
            clean.sum()
    def step(dbg_i=None):
        if graph is not None:
            graph.replay()
        else:
            moe.forward(x, y, wsp, st, dbg_i)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    L = wl.layers
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * L)] for _ in range(args.steps)]
    for evs in kev:            # torch creates CUDA events on first record
        for e in evs:
            e.record(stream)
    # per-kernel events force the one-launch-per-phase path: only used there
    kdbg = [None if (persistent or graph is not None) else moe.expert_timing(evs) for evs in kev]
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local, args.clocks_csv) if rank == 0 else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.1)
    t_wall = time.perf_counter()
    torch.cuda.profiler.start()   # a profiler started with --profile-from-start off sees the timed region only
    for i in range(args.steps):
        flush_l2(i)
        ev[i][0].record(stream)
        step(kdbg[i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    wall = time.perf_counter() - t_wall
    if ws > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.__exit__()
    per = [a.elapsed_time(b) * 1e3 for a, b in ev]   # us per forward
    if persistent or graph is not None:   # the whole forward is one kernel / one graph
        kern = [v / L for v in per]
    else:
        kern = [sum(evs[2 * l].elapsed_time(evs[2 * l + 1]) for l in range(L)) * 1e3 / L for evs in kev]
    us = statistics.mean(per)
    kern_us = statistics.mean(kern)
    # the same K steps under the other L2 protocol (not flushed <-> flushed clean), for reference
    other = "none" if args.flush != "none" else "clean"
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2(i, other)
        ev2[i][0].record(stream)
        step()
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    per2 = [a.elapsed_time(b) * 1e3 / wl.layers for a, b in ev2]
    l2_other = {"l2": FLUSH_DESC[other], "us_per_layer": round(statistics.mean(per2), 2),
                "dist_us_per_layer": _percentiles(per2)}
    st_code = pkg.moe_mxfp4_check(moe.handle, wsp.data_ptr(), st)
    if st_code != 0:
        raise pkg.MoeError(st_code, "forward")
    phases = None
    if persistent:   # CTA 0's phase-end timestamps of the last forward (workspace bytes 64..)
        nst = 2 + 4 * min(L, 8)
        ts = wsp[64:64 + 8 * nst].cpu().view(torch.int64).tolist()
        names = ["staging"] + [f"l{l}_{n}" for l in range(min(L, 8)) for n in ("router", "route", "experts", "combine")]
        phases = {n: round((ts[i + 1] - ts[i]) / 1e3, 2) for i, n in enumerate(names)}
        sub = wsp[64 + 8 * 34:64 + 8 * 55].cpu().view(torch.int64).tolist()   # routing / router sub-steps, layer 0
        phases["l0_route_steps"] = [round((sub[6 + i + 1] - sub[6 + i]) / 1e3, 2) for i in range(4)]
        phases["l0_router_unit0"] = [round((sub[14 + i + 1] - sub[14 + i]) / 1e3, 2) for i in range(4)]
        # CTA 0: its router units, the operand split, the wait at the barrier
        phases["l0_router_cta0"] = [round((sub[19] - ts[1]) / 1e3, 2), round((sub[20] - sub[19]) / 1e3, 2),
                                    round((ts[2] - sub[20]) / 1e3, 2)]
        if wl.T * wl.k > 64 or wl.T * wl.E > 8192:   # routed through the workspace: logits sum, top-k,
            # grouping (CTA 0), work list, operand gather (from the router phase's end)
            marks = [ts[2]] + sub[0:5]
            phases["l0_large_route_steps"] = [round((marks[i + 1] - marks[i]) / 1e3, 2) for i in range(5)]
    if ws > 1:
        t = torch.tensor([us], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        us = float(t.item())

    # end to end: host buffers through the C ABI, copies inside the timed region
    xh = inputs.x.clone().pin_memory()
    yh = torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory()
    for _ in range(3):
        moe.forward_host(xh, yh, wsp)
    e2e = []
    for i in range(args.steps):
        flush_l2(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        moe.forward_host(xh, yh, wsp)
        e2e.append((time.perf_counter() - t0) * 1e6)
    e2e_us = statistics.mean(e2e)

    if rank != 0:
        return
    peak, peak_kind = _peaks()
    gbs = alg_bytes / (us * 1e-6) / 1e9
    # algorithmic bytes of the timed kernel per layer: the persistent kernel moves all
    # of the layer's bytes; the separate expert kernel the routed experts' nibbles and scales
    kern_bytes = alg_bytes / wl.layers if (persistent or graph is not None) else \
        sum(n_active) * wl.expert_bytes / wl.layers
    kern_gbs = kern_bytes / (kern_us * 1e-6) / 1e9
    if persistent:
        launches_per_step = -(-wl.layers // 8)
    elif graph is not None:
        launches_per_step = (1 if wl.norm else 0) + 6 * wl.layers   # replayed inside one graph
    elif moe_tma(wl):
        launches_per_step = (1 if wl.norm else 0) + 6 * wl.layers
    else:
        launches_per_step = 1 + 5 * wl.layers + (wl.layers if wl.norm else 0)
    clocks = sampler.summary() if sampler else None
    line = {
        "metric": "us_per_moe_layer_per_verify_block", "value": round(us / wl.layers, 2), "unit": "us",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (MXFP4 weights)",
        "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "layers": wl.layers, "path": "persistent" if persistent else args.path,
                   "expert_layout": "packed" if packed else "canonical",
                   "routed_experts": n_active, "algorithmic_bytes": alg_bytes,
                   "l2": FLUSH_DESC[args.flush],
                   "parallelism": f"replicas{ws}"},
        "hbm_gbs": round(gbs, 1),
        "implied_tokens_per_s": round(ACCEPTANCE_LENGTH / (us * 1e-6), 1),
        "roofline": {"bound": "hbm", "achieved": round(kern_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(kern_gbs / peak, 4),
                     "frac_nominal": round(kern_gbs / NOMINAL_HBM_GBS, 4),
                     "traffic": layer_traffic(wl) if persistent else None, "peak_kind": peak_kind,
                     "kernel": "persistent forward kernel" if persistent else
                               "whole forward (CUDA graph of the per-phase launches)" if graph is not None else
                               "expert FFN kernel",
                     "kernel_us_per_layer": round(kern_us, 2),
                     "kernel_bytes_per_layer": int(kern_bytes)},
        "forward_hbm_frac": round(gbs / peak, 4),
        "forward_hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
        "l2_other_protocol": l2_other,
        "dist_us_per_layer": _percentiles([v / wl.layers for v in per]),
        "phases_us": phases,
        "e2e": {"value": round(e2e_us / wl.layers, 2), "unit": "us", "h2d_bytes_per_step": wl.T * wl.H * 2,
                "d2h_bytes_per_step": wl.T * wl.H * 4},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s": round(wall, 4),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line))


FLUSH_DESC = {
    "write": "flushed between steps: 256 MiB write outside the per-step events (leaves dirty lines)",
    "clean": "flushed between steps: 256 MiB write, then a 256 MiB read, outside the per-step events "
             "(cold, clean L2); inputs also larger than L2",
    "none": "not flushed: inputs larger than L2 -- every step streams the routed experts' weights "
            "(algorithmic_bytes, several times the 129 MB L2) from HBM; the kernel's code and a few KB of "
            "buffers stay in L2 as in a decode loop",
}


# the sources the persistent forward kernel is compiled from
KERNEL_SOURCES = ("common.cuh", "expert_tc.cuh", "moe_mxfp4.cu", "pack.cuh", "persist.cuh", "ptx.cuh", "route.cuh",
                  "worklist.cuh")


def kernel_sources_sha256():
    """Hash of the persistent kernel's sources (the same recipe as profiles/dram_traffic.json)."""
    import hashlib
    csrc = os.path.join(ROOT, "mxfp4_moe_expert_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in KERNEL_SOURCES]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes per launch of the timed kernel from the committed ncu capture of this
    workload, or None when there is none or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    e = json.load(open(p)).get(workload)
    if not e or e.get("source_sha256") != kernel_sources_sha256():
        return None
    return int(e["dram_read_bytes"] + e["dram_write_bytes"])


def layer_traffic(wl):
    """The captured DRAM bytes of one launch per layer it runs (a launch runs up to 8
    layers), on the same per-layer basis as `kernel_bytes_per_layer`; None without a
    current capture."""
    t = measured_traffic(wl.name)
    return None if t is None else int(round(t / min(wl.layers, 8)))


def _percentiles(v):
    """Median, 10th and 90th percentile (nearest rank) of the per-step times."""
    q = sorted(v)
    pick = lambda f: q[min(len(q) - 1, max(0, int(round(f * (len(q) - 1)))))]
    return {"median": round(statistics.median(q), 2), "p10": round(pick(0.1), 2), "p90": round(pick(0.9), 2)}


def run_sweep(args):
    """Multi-stream sweep: the 384-expert layer over verify blocks of
    8 x {1, 4, 16, 32, 64} tokens (streams of 8 positions), persistent forward, clean L2
    before each step.  Prints one JSON line with a row per block size."""
    import torch

    import mxfp4_moe_expert_gb300 as pkg
    from mxfp4_moe_expert_gb300.synth import WORKLOADS, make_inputs
    from mxfp4_moe_expert_gb300.workload import device_layers, touched_bytes

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    base = WORKLOADS["large"]
    sizes = [8, 32, 128, 256, 512]
    _, layers = device_layers(base, device=dev, packed=args.layout == "packed")
    moe = pkg.MoeLayers(hidden=base.H, inter=base.I, num_experts=base.E, top_k=base.k, max_tokens=max(sizes),
                        layers=layers)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = stream.cuda_stream
    peak, peak_kind = _peaks()
    rows = []
    for T in sizes:
        wl = base.scaled(T=T, name=f"large_T{T}")
        x = make_inputs(wl).x.to(dev)
        y = torch.empty((T, base.H), dtype=torch.float32, device=dev)
        wsp = moe.new_workspace(T, dev)
        bufs, dbg = moe.debug_buffers(T, dev)
        moe.forward(x, y, wsp, st, dbg, check=True)
        counts = bufs["expert_counts"].cpu()
        alg = touched_bytes(wl, [counts[0]])
        chunks = int(((counts[0] + 7) // 8).sum())
        for _ in range(max(args.warmup, 3)):
            moe.forward(x, y, wsp, st)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            clean.sum()
            ev[i][0].record(stream)
            moe.forward(x, y, wsp, st)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        assert pkg.moe_mxfp4_check(moe.handle, wsp.data_ptr(), st) == 0
        us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev)
        rows.append({"tokens": T, "streams": T // 8, "us_per_forward": round(us, 2),
                     "us_per_stream": round(us / (T // 8), 2), "routed_experts": int((counts[0] > 0).sum()),
                     "chunks": chunks, "algorithmic_bytes": alg, "hbm_gbs": round(alg / (us * 1e-6) / 1e9, 1),
                     "frac_of_peak": round(alg / (us * 1e-6) / 1e9 / peak, 4)})
        del wsp, bufs
    print(json.dumps({"metric": "multi_stream_sweep", "unit": "us", "config": {"workload": "large", "H": base.H,
                      "I": base.I, "E": base.E, "k": base.k, "path": "persistent", "expert_layout": args.layout,
                      "l2": FLUSH_DESC["clean"]}, "peak_gbs": peak, "peak_kind": peak_kind,
                      "steps": args.steps, "rows": rows}))


def moe_tma(wl):
    """The forward runs the TMA expert kernel (7 launches per layer, plus the
    input staging) when H and I are multiples of 512; else the multi-kernel path."""
    return wl.H % 512 == 0 and wl.I % 512 == 0 and wl.T * wl.k <= 4096


def cpu_baseline(wl):
    """The oracle on the host cores (OracleHost): one warm-up and one timed forward of the
    whole verify block, every routed expert evaluated."""
    host = OracleHost(wl)
    try:
        host.forward()
        t0 = time.perf_counter()
        host.forward()
        dt = time.perf_counter() - t0
    finally:
        host.close()
    return {"value": round(dt * 1e6 / wl.layers, 1), "unit": "us", "cores": host.n, "kind": "oracle",
            "sample": f"the whole verify block: all {sum(host.routed)} routed experts, no sampling "
                      f"({host.n} worker processes)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="large", choices=["tiny", "mid", "large", "batched", "stack"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default="", help="keep the nvidia-smi clock samples of the timed region here")
    ap.add_argument("--flush", default="none", choices=["write", "clean", "none"],
                    help="L2 state before each timed step (see FLUSH_DESC); the line also carries the same "
                         "steps under the other protocol (none <-> clean)")
    ap.add_argument("--path", default="persistent", choices=["persistent", "multi", "graph"],
                    help="one cooperative launch per forward, one launch per phase, or those launches "
                         "captured in a CUDA graph")
    ap.add_argument("--sweep", action="store_true", help="multi-stream sweep of the 384-expert layer")
    ap.add_argument("--layout", default="packed", choices=["packed", "canonical"],
                    help="expert weights streamed from the packed (tile-major) copy or the canonical layout")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling aid: the workload with this many experts (a reduced layer for ncu captures "
                         "that must hold a few GB at most); the line names it <workload>_E<n>")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
