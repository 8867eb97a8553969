"""The persistent forward's state section stays at rest between forwards.

Every launch of the persistent kernel returns the counters, flags and grid-barrier word
at the start of the workspace to rest (zero), so the next forward on that workspace is a
single kernel launch with no clearing copy before it.  These tests run many forwards on
one workspace without reading the status in between -- blocks routed in shared memory and
blocks routed through the workspace (they use different counters), and a stack deeper
than one launch -- and require every output to equal, bit for bit, the output of a
forward on a freshly zeroed workspace.  They also overwrite the state tag, to check that a
forward on a workspace changed behind the library's back records MOE_ERR_WORKSPACE and
does nothing, and that reading the error brings the section back to rest; and they check
that an error stays until it is read: a forward issued behind a timed-out one does
nothing and returns at once.
"""
import os

import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from mxfp4_moe_expert_gb300.synth import Workload
from mxfp4_moe_expert_gb300.workload import device_layers

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()


def _moe(wl, layers, flags=0, **kw):
    if wl.norm:
        flags |= pkg.MOE_FLAG_NORM
    return pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T,
                         layers=layers, flags=flags, rms_eps=wl.rms_eps, **kw)


def _fresh(moe, x):
    """Output of a forward on a workspace of its own (zeroed by the library on first use)."""
    ws = moe.new_workspace(moe.cfg.max_tokens, x.device)
    y = moe.forward(x, workspace=ws, check=True)
    torch.cuda.synchronize()
    return y


def test_many_forwards_on_one_workspace_with_both_block_kinds():
    # 40 tokens x top-4 = 160 pairs: routed through the workspace; 8 x 4 = 32 pairs: in shared memory
    wl = Workload("state_mixed", T=40, H=1024, I=512, E=16, k=4, seed=0x5EED0300)
    inputs, layers = device_layers(wl, device=DEV)
    moe = _moe(wl, layers)
    x = inputs.x.to(DEV)
    blocks = {40: x, 8: x[:8].contiguous(), 3: x[3:6].contiguous()}
    ref = {T: _fresh(moe, xb) for T, xb in blocks.items()}
    ws = moe.new_workspace(wl.T, DEV)
    order = [40, 8, 8, 40, 3, 40, 40, 8, 3, 3, 40, 8]
    outs = [moe.forward(blocks[T], workspace=ws) for T in order]   # no status read in between
    assert pkg.moe_mxfp4_check(moe.handle, ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == pkg.MOE_OK
    for i, (T, y) in enumerate(zip(order, outs)):
        assert torch.equal(y, ref[T]), (i, T)
    moe.close()


def test_stack_deeper_than_one_launch_reuses_its_workspace():
    """Ten layers take two launches per forward (eight layers per launch); both leave
    the section at rest for the launch after them."""
    wl = Workload("state_stack10", T=8, H=1024, I=512, E=8, k=2, layers=10, norm=True, seed=0x5EED0301)
    inputs, layers = device_layers(wl, device=DEV)
    moe = _moe(wl, layers)
    x = inputs.x.to(DEV)
    ref = _fresh(moe, x)
    ws = moe.new_workspace(wl.T, DEV)
    outs = [moe.forward(x, workspace=ws) for _ in range(5)]
    assert pkg.moe_mxfp4_check(moe.handle, ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == pkg.MOE_OK
    for i, y in enumerate(outs):
        assert torch.equal(y, ref), i
    moe.close()


def test_overwritten_state_tag_is_reported_then_recovered():
    wl = Workload("state_tag", T=8, H=1024, I=512, E=16, k=4, seed=0x5EED0302)
    inputs, layers = device_layers(wl, device=DEV)
    moe = _moe(wl, layers)
    x = inputs.x.to(DEV)
    ref = _fresh(moe, x)
    st = torch.cuda.current_stream().cuda_stream
    ws = moe.new_workspace(wl.T, DEV)
    assert torch.equal(moe.forward(x, workspace=ws, check=True), ref)
    ws[32:40] = 0xA5                                     # the state tag, changed behind the library's back
    y = torch.full((wl.T, wl.H), float("nan"), device=DEV)
    moe.forward(x, y=y, workspace=ws)
    assert pkg.moe_mxfp4_check(moe.handle, ws.data_ptr(), st) == pkg.MOE_ERR_WORKSPACE
    assert torch.isnan(y).all()                          # the forward did nothing
    assert pkg.moe_mxfp4_check(moe.handle, ws.data_ptr(), st) == pkg.MOE_OK   # reading it restored the section
    assert torch.equal(moe.forward(x, workspace=ws, check=True), ref)
    moe.close()


def test_error_stays_until_read_and_later_forwards_do_nothing():
    """A grid-barrier arrival withheld on purpose (MOE_FLAG_DEBUG_STALL) makes the waits
    run out after 20 ms; the next forward on that workspace finds the abort flag and
    leaves at once, without touching y; the error is still there when it is read."""
    wl = Workload("state_sticky", T=8, H=1024, I=512, E=16, k=4, seed=0x5EED0303)
    inputs, layers = device_layers(wl, device=DEV)
    x = inputs.x.to(DEV)
    good = _moe(wl, layers)
    ref = _fresh(good, x)
    stalled = _moe(wl, layers, flags=pkg.MOE_FLAG_DEBUG_STALL, timeout_us=20000)
    st = torch.cuda.current_stream().cuda_stream
    ws = stalled.new_workspace(wl.T, DEV)
    stalled.forward(x, workspace=ws)                     # times out on the device
    y = torch.full((wl.T, wl.H), float("nan"), device=DEV)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    stalled.forward(x, y=y, workspace=ws)
    t1.record()
    torch.cuda.synchronize()
    assert t0.elapsed_time(t1) < 5.0                     # ms: no 20 ms wait, it left at once
    assert torch.isnan(y).all()
    assert pkg.moe_mxfp4_check(stalled.handle, ws.data_ptr(), st) == pkg.MOE_ERR_TIMEOUT
    # another handle on the same workspace zeroes the section first and runs normally
    assert torch.equal(good.forward(x, workspace=ws, check=True), ref)
    stalled.close()
    good.close()
