"""Every packed weight byte decodes on the device as the MXFP4 format defines.

An expert layer whose E2M1 bytes run through all 256 values in every row (so every
code sits in both the low and the high nibble, next to every other code), with
varied E8M0 scales, goes through the persistent tensor-core forward and the
one-launch-per-phase forward; both are compared with the fp64 oracle, whose decode is
pinned to the format's value table by the CPU tests.  A wrong code value, a swapped
nibble order or a scale applied to the wrong 32-element block breaks the tolerance.
"""
import numpy as np
import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from mxfp4_moe_expert_gb300.synth import Workload, make_inputs
from mxfp4_moe_expert_gb300.workload import alloc_layer
from oracle import moe_oracle as O
from parity_util import assert_rows_close, bf16_np, oracle_layer_args

pytestmark = pytest.mark.gpu

DEV = "cuda"
WL = Workload("all_bytes", T=8, H=512, I=512, E=4, k=2, seed=0x5EED0130)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()


def _crafted_bytes(wl):
    """Per matrix: q[e, r, c] = (37 (e rows + r) + c) mod 256 over the row's K / 2 = 256
    bytes (each byte value once per row), and scale bytes 121..125 (|w| <= 6 / 16)."""
    rng = np.random.default_rng(0x5EED)
    out = {}
    for m, (rows, K) in {"gate": (wl.I, wl.H), "up": (wl.I, wl.H), "down": (wl.H, wl.I)}.items():
        r = np.arange(wl.E * rows, dtype=np.int64)[:, None]
        c = np.arange(K // 2, dtype=np.int64)[None, :]
        q = ((37 * r + c) % 256).astype(np.uint8).reshape(wl.E, rows, K // 2)
        s = rng.integers(121, 126, size=(wl.E, rows, K // 32)).astype(np.uint8)
        out[m] = (q, s)
    return out


@pytest.mark.parametrize("flags,packed,T", [(0, False, 8), (pkg.MOE_FLAG_MULTI_KERNEL, False, 8), (0, True, 8),
                                            (pkg.MOE_FLAG_MULTI_KERNEL, True, 8), (0, True, 40),
                                            (pkg.MOE_FLAG_NO_DENSE, True, 40)],
                         ids=["persistent", "multi_kernel", "persistent_packed", "multi_kernel_packed",
                              "persistent_dense", "persistent_gathered_8x8"])
def test_every_weight_byte_decodes_as_the_format_defines(flags, packed, T):
    """T = 40 (80 pairs) is routed through the workspace: its chunks take the dense operand
    (32 pairs x 4 terms), or 16 pairs x 8 terms with MOE_FLAG_NO_DENSE."""
    wl = WL.scaled(T=T)
    assert (wl.H // 2) == 256 and (wl.I // 2) == 256   # one full byte cycle per row
    inputs = make_inputs(wl)
    crafted = _crafted_bytes(wl)
    for m in ("gate", "up", "down"):
        q = crafted[m][0]
        assert all(len(np.unique(q[e, r])) == 256 for e in range(wl.E) for r in (0, q.shape[1] - 1))
    L = alloc_layer(wl, DEV)
    for m, (q, s) in crafted.items():
        L[m + "_q"].copy_(torch.from_numpy(q))
        L[m + "_s"].copy_(torch.from_numpy(s))
    lt = inputs.layers[0]
    L["router_w"] = lt.router_w.to(DEV).contiguous()
    L["router_b"] = lt.router_b.to(DEV).contiguous()
    L["norm_w"] = None
    if packed:   # the experts are read from the packed copy only
        L["packed"] = pkg.pack(L, wl.H, wl.I, wl.E)
        for m in ("gate", "up", "down"):
            L[m + "_q"] = L[m + "_s"] = None
    moe = pkg.MoeLayers(hidden=wl.H, inter=wl.I, num_experts=wl.E, top_k=wl.k, max_tokens=wl.T, layers=[L],
                        flags=flags)
    bufs, dbg = moe.debug_buffers(wl.T)
    y = moe.forward(inputs.x.to(DEV), dbg=dbg, check=True)
    torch.cuda.synchronize()

    wr, b, _ = oracle_layer_args(inputs, 0)
    ref = O.moe_layer(bf16_np(inputs.x), wr, b, wl.k,
                      lambda e: O.ExpertMatrices(crafted["gate"][0][e], crafted["gate"][1][e], crafted["up"][0][e],
                                                 crafted["up"][1][e], crafted["down"][0][e], crafted["down"][1][e]))
    assert np.array_equal(bufs["topk_idx"][0].cpu().numpy(), ref["idx"])
    assert np.array_equal(bufs["perm"][0].cpu().numpy(), ref["perm"])
    assert_rows_close(y.double().cpu().numpy(), ref["y"], what="all bytes")
    moe.close()


def test_packed_layout_is_the_documented_tile_order():
    """moe_mxfp4_pack against the layout stated in include/moe_mxfp4.h, rebuilt here with
    numpy from random canonical bytes: code tiles of 256 rows x 128 B (gate rows then the
    same up rows, or 256 down rows) per 256-K stage, scale groups of 256 rows x 8 G B,
    three 256-byte-aligned sections."""
    wl = Workload("pack", T=1, H=1536, I=1024, E=3, k=1, seed=0)
    rng = np.random.default_rng(3)
    L, canon = {}, {}
    for m, (rows, K) in {"gate": (wl.I, wl.H), "up": (wl.I, wl.H), "down": (wl.H, wl.I)}.items():
        q = rng.integers(0, 256, size=(wl.E, rows, K // 2), dtype=np.uint8)
        sc = rng.integers(0, 255, size=(wl.E, rows, K // 32), dtype=np.uint8)
        canon[m] = (q, sc)
        L[m + "_q"] = torch.from_numpy(q).to(DEV)
        L[m + "_s"] = torch.from_numpy(sc).to(DEV)
    got = pkg.pack(L, wl.H, wl.I, wl.E).cpu().numpy()
    E, H, I = wl.E, wl.H, wl.I

    def group(K):
        return next(g for g in (8, 6, 4, 2) if (K // 256) % g == 0)

    def tiles(a, b, K, width):
        """[E, rows, K/width] canonical -> [E][blocks][K/width/w][256 rows][w] with w = 128 (codes)
        or 8 G (scales); a and b give rows 0..127 and 128..255 of a tile (gate / up), or b is
        None and a tile is 256 consecutive rows of a."""
        w = 128 if width == 2 else 8 * group(K)
        cols = a.shape[2]
        if b is None:
            t = a.reshape(E, a.shape[1] // 256, 256, cols // w, w)
        else:
            t = np.stack([a.reshape(E, a.shape[1] // 128, 128, cols // w, w),
                          b.reshape(E, b.shape[1] // 128, 128, cols // w, w)], axis=2)
            t = t.reshape(E, a.shape[1] // 128, 256, cols // w, w)
        return np.ascontiguousarray(t.transpose(0, 1, 3, 2, 4)).reshape(-1)

    sections = [np.concatenate([tiles(canon["gate"][0], canon["up"][0], H, 2),
                                tiles(canon["down"][0], None, I, 2)]),
                tiles(canon["gate"][1], canon["up"][1], H, 32),
                tiles(canon["down"][1], None, I, 32)]
    off = 0
    st, n = pkg.moe_mxfp4_packed_bytes(wl.H, wl.I, wl.E)
    for sec in sections:
        assert np.array_equal(got[off:off + sec.size], sec), off
        off = (off + sec.size + 255) // 256 * 256
    assert st == pkg.MOE_OK and n == off == got.size
