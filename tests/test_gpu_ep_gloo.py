"""Expert parallelism with the library's own partials: two ranks (processes) each run the
layer on their expert range through the C ABI on the GPU, and the decomposition's one
exchange step -- an all-reduce sum of the ranks' partial y -- runs over gloo on the host.
The sum must equal the fp64 oracle's full layer on every row.  Every run here has one GPU,
so both ranks share it; their kernels never wait on each other (the only exchange is the
host-side all-reduce after each rank's forward has finished)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

WL_ARGS = dict(name="ep_two_ranks", T=13, H=1024, I=512, E=16, k=4, seed=0x5EED0400)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import mxfp4_moe_expert_gb300 as pkg
        from mxfp4_moe_expert_gb300.shard import expert_ranges
        from mxfp4_moe_expert_gb300.synth import Workload
        from mxfp4_moe_expert_gb300.workload import device_layers
        from parity_util import oracle_quantizer_to
        pkg.load_library()
        wl = Workload(**WL_ARGS)
        inputs, layers = device_layers(wl, device="cuda", weights_device="cpu", quantizer=oracle_quantizer_to("cuda"))
        # contiguous expert ranges balanced by the bytes each expert would move (every expert here)
        lo, hi = expert_ranges(wl.E, world, [float(wl.expert_bytes)] * wl.E)[rank]
        moe = pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T,
                            layers=layers, expert_begin=lo, expert_end=hi)
        part = moe.forward(inputs.x.to("cuda"), check=True).cpu()
        moe.close()
        y = part.clone()
        dist.all_reduce(y, op=dist.ReduceOp.SUM)   # the exchange step, on the ranks' CUDA-produced partials
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y.double().numpy())
        np.save(os.path.join(out_dir, f"part{rank}.npy"), part.double().numpy())
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_library_partials_allreduce_to_the_oracle_layer(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import mxfp4_moe_expert_gb300 as pkg
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    from mxfp4_moe_expert_gb300.synth import Workload, make_inputs
    from oracle import moe_oracle as O
    from parity_util import OracleExperts, assert_rows_close, bf16_np, oracle_layer_args

    world = 2
    mp.start_processes(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    wl = Workload(**WL_ARGS)
    inputs = make_inputs(wl)
    x = bf16_np(inputs.x)
    wr, b, _ = oracle_layer_args(inputs, 0)
    full = O.moe_layer(x, wr, b, wl.k, OracleExperts(wl, 0))["y"]
    ys = [np.load(tmp_path / f"y{r}.npy") for r in range(world)]
    parts = [np.load(tmp_path / f"part{r}.npy") for r in range(world)]
    assert np.array_equal(ys[0], ys[1])                       # every rank holds the same sum
    assert not np.array_equal(parts[0], parts[1])             # each rank computed its own shard
    assert_rows_close(ys[0], full, what="two-rank expert parallel")
