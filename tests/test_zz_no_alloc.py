"""The allocation-free forward gives the same layer output as the workspace forward.

moe_mxfp4_forward_static is for callers that cannot allocate device memory when
they run the layer (a host program that pre-reserved all of HBM for its own pool,
a plugin whose host framework owns every device allocation, a latency-bound loop
that cannot afford an allocation's device-wide synchronisation).  It keeps its
workspace in a fixed array inside the library.  This file is named so that pytest
collects it last; it sets up everything it uses, so it also passes alone.
"""
import os

import numpy as np
import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from mxfp4_moe_expert_gb300.synth import Workload
from mxfp4_moe_expert_gb300.workload import device_layers
from parity_util import assert_rows_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()
    wl = Workload("no_alloc", T=13, H=1024, I=512, E=16, k=4, seed=0x5EED0200)
    inputs, layers = device_layers(wl, device="cuda")
    moe = pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T, layers=layers)
    yield wl, inputs, layers, moe
    moe.close()


def test_static_workspace_forward_matches_workspace_forward_twice(layer):
    wl, inputs, layers, moe = layer
    x = inputs.x.to("cuda")
    ref = moe.forward(x, check=True).double().cpu().numpy()
    st = torch.cuda.current_stream().cuda_stream
    for call in range(2):   # the second call reuses the array the first one left behind
        y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
        status = pkg.moe_mxfp4_forward_static(moe.handle, x.data_ptr(), wl.T, y.data_ptr(), st)
        assert status == pkg.MOE_OK, pkg.moe_mxfp4_status_string(status)
        got = y.double().cpu().numpy()
        assert np.isfinite(got).all(), call
        assert_rows_close(got, ref, what=f"static call {call}")


def test_static_workspace_forward_on_a_larger_block_twice():
    """A block of 24 tokens x top-4 (96 pairs) is routed through the workspace and its
    input operand is gathered per chunk: the sections of the array that the small
    block above leaves unused are written and read here, on two calls in a row."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = Workload("no_alloc_larger", T=24, H=1024, I=512, E=12, k=4, seed=0x5EED0201)
    inputs, layers = device_layers(wl, device="cuda")
    moe = pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T, layers=layers)
    assert wl.T * wl.k > 64 and moe.workspace_bytes(wl.T) <= pkg.MOE_MXFP4_STATIC_WORKSPACE_BYTES
    x = inputs.x.to("cuda")
    ref = moe.forward(x, check=True).double().cpu().numpy()
    st = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
        status = pkg.moe_mxfp4_forward_static(moe.handle, x.data_ptr(), wl.T, y.data_ptr(), st)
        assert status == pkg.MOE_OK, pkg.moe_mxfp4_status_string(status)
        got = y.double().cpu().numpy()
        assert np.isfinite(got).all(), call
        assert_rows_close(got, ref, what=f"static call {call} (larger block)")
    moe.close()


def test_static_workspace_rejects_sizes_beyond_its_limit(layer):
    wl, inputs, layers, _ = layer
    big = Workload("no_alloc_big", T=1024, H=wl.H, I=wl.I, E=wl.E, k=wl.k, seed=wl.seed)
    moe = pkg.MoeLayers(hidden=big.H, inter=big.I, num_experts=big.E, top_k=big.k, max_tokens=big.T, layers=layers)
    assert moe.workspace_bytes(big.T) > pkg.MOE_MXFP4_STATIC_WORKSPACE_BYTES
    x = torch.zeros((big.T, big.H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((big.T, big.H), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert pkg.moe_mxfp4_forward_static(moe.handle, x.data_ptr(), big.T, y.data_ptr(), st) == pkg.MOE_ERR_WORKSPACE
    assert not y.any()
    moe.close()
