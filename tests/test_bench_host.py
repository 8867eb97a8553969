"""Host-side arithmetic of the measurement (CPU only): the algorithmic bytes the
roofline divides by, and the per-step statistics of the bench line."""
import importlib.util
import os

import pytest

from mxfp4_moe_expert_gb300.synth import WORKLOADS
from mxfp4_moe_expert_gb300.workload import touched_bytes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_expert_bytes_is_three_mxfp4_matrices():
    # 3 H x I matrices of 4-bit codes plus one E8M0 byte per 32 codes: 0.53125 B per weight
    wl = WORKLOADS["large"]
    assert wl.expert_bytes == 3 * wl.H * wl.I * 17 // 32 == 23_396_352


def test_touched_bytes_of_the_384_expert_layer():
    # 60 routed experts + bf16 router + fp32 bias + bf16 x read + fp32 y written
    wl = WORKLOADS["large"]
    counts = [0] * wl.E
    for e in range(60):
        counts[e * 6] = 1
    want = 60 * 23_396_352 + 384 * 7168 * 2 + 384 * 4 + 8 * 7168 * 2 + 8 * 7168 * 4
    assert touched_bytes(wl, [counts]) == want == 1_409_631_744


def test_touched_bytes_of_a_stack_counts_every_layer_once():
    wl = WORKLOADS["stack"]
    per_layer = [[1 if e < 10 else 0 for e in range(wl.E)] for _ in range(wl.layers)]
    layer = 10 * wl.expert_bytes + wl.E * wl.H * 2 + wl.E * 4 + wl.H * 2
    assert touched_bytes(wl, per_layer) == wl.layers * layer + wl.T * wl.H * 6


def test_percentiles_nearest_rank():
    b = _bench()
    d = b._percentiles([5.0, 1.0, 2.0, 3.0, 4.0, 6.0, 7.0, 8.0, 9.0, 10.0])
    assert d == {"median": 5.5, "p10": 2.0, "p90": 9.0}
    assert b._percentiles([3.0]) == {"median": 3.0, "p10": 3.0, "p90": 3.0}


def test_tma_path_rule():
    b = _bench()
    assert b.moe_tma(WORKLOADS["large"]) and b.moe_tma(WORKLOADS["batched"])
    assert not b.moe_tma(WORKLOADS["tiny"])   # H = 256: the one-launch-per-phase path


@pytest.mark.parametrize("name", ["large", "mid", "batched", "stack"])
def test_traffic_record_names_a_summary_and_a_source_hash(name):
    import json
    rec = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))[name]
    assert rec["dram_read_bytes"] > 0 and rec["dram_write_bytes"] > 0
    assert len(rec["source_sha256"]) == 64


def test_traffic_records_are_keyed_to_the_current_kernel_sources():
    """The committed DRAM counters describe the kernel as built from these sources (the bench
    reports them only then): a kernel change without a new capture shows up here."""
    import json
    recs = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    h = _bench().kernel_sources_sha256()
    assert all(recs[w]["source_sha256"] == h for w in ("large", "mid", "batched", "stack"))


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line with
    the keys the driver reads; run on the small workload so it takes a second."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us" and d["higher_is_better"] is False
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0   # at least 3 warm-up steps, whatever asked
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches N > 1 (torchrun, one process per rank), rank 0
    alone prints the reference line and the other rank exits 0 without work."""
    import json
    import socket
    import subprocess
    import sys
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
