"""Device-resident layers for a seeded workload.

Draws the inputs of a workload with `synth` and MXFP4-encodes the expert
weights expert by expert with the library's CUDA quantizer (or a quantizer the
caller passes), into [E, rows, cols/2] nibble and [E, rows, cols/32] scale
tensors that stay resident in HBM.
"""
from __future__ import annotations

import torch

from . import pack as _pack
from . import quantize as _cuda_quantize
from .synth import Inputs, Workload, expert_weight, make_inputs


def alloc_layer(wl: Workload, device) -> dict:
    E, H, I = wl.E, wl.H, wl.I
    u8 = dict(dtype=torch.uint8, device=device)
    return dict(
        gate_q=torch.empty((E, I, H // 2), **u8), gate_s=torch.empty((E, I, H // 32), **u8),
        up_q=torch.empty((E, I, H // 2), **u8), up_s=torch.empty((E, I, H // 32), **u8),
        down_q=torch.empty((E, H, I // 2), **u8), down_s=torch.empty((E, H, I // 32), **u8),
    )


def device_layers(wl: Workload, inputs: Inputs | None = None, device="cuda", weights_device=None,
                  quantizer=None, packed=False) -> tuple[Inputs, list]:
    """Returns (inputs, layers): layers[l] is a dict of device tensors accepted by MoeLayers.

    weights_device: where the fp32 master weights are drawn (default: `device`).
    quantizer(w_fp32) -> (q, s) tensors; default: the library's CUDA kernel.
    packed: also add each layer's experts in the packed layout (layers[l]["packed"],
    made by moe_mxfp4_pack from the canonical tensors, which stay in the dict); the
    forward then streams the experts from the packed copy.
    """
    inputs = inputs or make_inputs(wl)
    weights_device = weights_device or device
    layers = []
    for l in range(wl.layers):
        L = alloc_layer(wl, device)
        for e in range(wl.E):
            for m in ("gate", "up", "down"):
                w = expert_weight(wl, l, e, m, weights_device)
                if quantizer is None:
                    q, s = _cuda_quantize(w.to(device).contiguous())
                else:
                    q, s = quantizer(w)
                L[m + "_q"][e].copy_(q)
                L[m + "_s"][e].copy_(s)
                del w
        lt = inputs.layers[l]
        L["router_w"] = lt.router_w.to(device).contiguous()
        L["router_b"] = lt.router_b.to(device).contiguous()
        L["norm_w"] = lt.norm_w.to(device).contiguous() if lt.norm_w is not None else None
        if packed:
            L["packed"] = _pack(L, wl.H, wl.I, wl.E)
        layers.append(L)
    return inputs, layers


def touched_bytes(wl: Workload, counts_per_layer) -> int:
    """Unique bytes one forward must move: the routed experts' nibbles and scales,
    router weights and bias, norm weights, x read (bf16) and y written (fp32)."""
    total = 0
    for counts in counts_per_layer:
        active = int((torch.as_tensor(counts) > 0).sum())
        total += active * wl.expert_bytes + wl.E * wl.H * 2 + wl.E * 4
        if wl.norm:
            total += wl.H * 2
    total += wl.T * wl.H * (2 + 4)
    return total


def repack(layers: list, wl: Workload) -> None:
    """(Re)makes layers[l]["packed"] from the canonical tensors of every layer (after
    the caller changed some expert bytes)."""
    for L in layers:
        L.pop("packed", None)
        L["packed"] = _pack(L, wl.H, wl.I, wl.E)
