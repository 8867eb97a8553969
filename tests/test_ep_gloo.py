"""Expert parallelism on the host, CPU only: the expert-range partition and the one
exchange step of the decomposition (an all-reduce sum of the ranks' partial y),
run as two gloo ranks over the fp64 oracle.  The GPU side of a shard (a layer
config with an expert range) is covered by the GPU parity tests; every box here
has one GPU, so the collective itself is exercised on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mxfp4_moe_expert_gb300.shard import expert_ranges
from mxfp4_moe_expert_gb300.synth import WORKLOADS, make_inputs
from oracle import moe_oracle as O
from parity_util import OracleExperts, bf16_np, oracle_layer_args


def _brute_force_ranges(cost, world):
    """Smallest possible max range cost, by trying every split (tiny inputs)."""
    n = len(cost)
    best = None

    def rec(start, left, cur):
        nonlocal best
        if left == 1:
            m = max(cur, sum(cost[start:]))
            best = m if best is None else min(best, m)
            return
        for end in range(start, n + 1):
            rec(end, left - 1, max(cur, sum(cost[start:end])))

    rec(0, world, 0.0)
    return best


def _check_partition(r, n, world):
    assert len(r) == world
    assert r[0][0] == 0 and r[-1][1] == n
    for (b0, e0), (b1, e1) in zip(r, r[1:]):
        assert e0 == b1 and b0 <= e0
    assert all(b <= e for b, e in r)


@pytest.mark.parametrize("n,world", [(8, 2), (7, 3), (5, 5), (3, 4), (0, 2), (12, 1)])
def test_expert_ranges_uniform(n, world):
    r = expert_ranges(n, world)
    _check_partition(r, n, world)
    sizes = [e - b for b, e in r]
    assert max(sizes) == -(-n // world)


def test_expert_ranges_match_brute_force_on_skewed_costs():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 9))
        world = int(rng.integers(1, 5))
        cost = [float(v) for v in rng.zipf(1.3, size=n).clip(max=50)]
        r = expert_ranges(n, world, cost)
        _check_partition(r, n, world)
        worst = max(sum(cost[b:e]) for b, e in r)
        assert worst == pytest.approx(_brute_force_ranges(cost, world)), (cost, world, r)


def test_expert_ranges_rejects_bad_arguments():
    with pytest.raises(ValueError):
        expert_ranges(4, 0)
    with pytest.raises(ValueError):
        expert_ranges(3, 2, [1.0, 2.0])
    with pytest.raises(ValueError):
        expert_ranges(2, 2, [1.0, -1.0])


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ep_rank(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = WORKLOADS["tiny"]
        inputs = make_inputs(wl)
        x = bf16_np(inputs.x)
        wr, b, _ = oracle_layer_args(inputs, 0)
        experts = OracleExperts(wl, 0)
        # expected touched bytes per expert from this block's routing: balance by bytes
        idx, _ = O.topk_gates(O.router_logits(x, wr, b), wl.k)
        counts = np.bincount(idx.reshape(-1), minlength=wl.E)
        cost = [float(c > 0) * wl.expert_bytes for c in counts]
        lo, hi = expert_ranges(wl.E, world, cost)[rank]

        class Zero:   # an expert outside this rank's range contributes nothing here
            def ffn(self, xrow):
                return np.zeros(wl.H)

        part = O.moe_layer(x, wr, b, wl.k, lambda e: experts(e) if lo <= e < hi else Zero())["y"]
        y = torch.from_numpy(np.ascontiguousarray(part))
        dist.all_reduce(y, op=dist.ReduceOp.SUM)   # the exchange step of expert parallelism
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y.numpy())
        np.save(os.path.join(out_dir, f"part{rank}.npy"), part)
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_allreduce_equals_full_layer(tmp_path):
    world = 2
    mp.start_processes(_ep_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    wl = WORKLOADS["tiny"]
    inputs = make_inputs(wl)
    x = bf16_np(inputs.x)
    wr, b, _ = oracle_layer_args(inputs, 0)
    full = O.moe_layer(x, wr, b, wl.k, OracleExperts(wl, 0))["y"]
    parts = [np.load(tmp_path / f"part{r}.npy") for r in range(world)]
    assert all(np.any(p != 0) for p in parts), "both ranks own routed experts"
    for r in range(world):
        y = np.load(tmp_path / f"y{r}.npy")
        np.testing.assert_allclose(y, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
