"""MXFP4 Mixture-of-Experts expert layer for GB300 (sm_103a).

Thin ctypes binding of the C ABI in include/moe_mxfp4.h: the functions below
carry the C names and only marshal arguments; every step of the layer runs in
the library's CUDA kernels.  PyTorch is used by callers for device memory and
streams only.  Importing this package does not load the library; the first
call does, and raises if the built library is missing (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmoe_mxfp4.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_CUDA = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_BAD_SCALE = -5
MOE_ERR_WORKSPACE = -6

MOE_FLAG_NORM = 1 << 0
MOE_FLAG_OUT_BF16 = 1 << 1
MOE_FLAG_MULTI_KERNEL = 1 << 2
MOE_FLAG_NO_DENSE = 1 << 3
MOE_FLAG_DEBUG_STALL = 1 << 4
MOE_FLAG_TRACE = 1 << 5

EXPORTED = (
    "moe_mxfp4_create",
    "moe_mxfp4_workspace_bytes",
    "moe_mxfp4_forward",
    "moe_mxfp4_forward_host",
    "moe_mxfp4_check",
    "moe_mxfp4_destroy",
    "moe_mxfp4_status_string",
    "moe_mxfp4_quantize",
    "moe_mxfp4_forward_static",
    "moe_mxfp4_accept",
    "moe_mxfp4_packed_bytes",
    "moe_mxfp4_pack",
    "moe_mxfp4_split_terms",
)

MOE_MXFP4_STATIC_WORKSPACE_BYTES = 16 << 20


class moe_mxfp4_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32),
        ("rms_eps", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("expert_begin", ctypes.c_int32),
        ("expert_end", ctypes.c_int32),
        ("timeout_us", ctypes.c_int32),
    ]


class moe_mxfp4_layer(ctypes.Structure):
    _fields_ = [
        ("router_w_dev", ctypes.c_void_p),
        ("router_b_dev", ctypes.c_void_p),
        ("gate_q_dev", ctypes.c_void_p),
        ("gate_s_dev", ctypes.c_void_p),
        ("up_q_dev", ctypes.c_void_p),
        ("up_s_dev", ctypes.c_void_p),
        ("down_q_dev", ctypes.c_void_p),
        ("down_s_dev", ctypes.c_void_p),
        ("norm_w_dev", ctypes.c_void_p),
        ("packed_dev", ctypes.c_void_p),
    ]


class moe_mxfp4_debug(ctypes.Structure):
    _fields_ = [
        ("topk_idx_dev", ctypes.c_void_p),
        ("topk_gate_dev", ctypes.c_void_p),
        ("expert_counts_dev", ctypes.c_void_p),
        ("expert_offsets_dev", ctypes.c_void_p),
        ("perm_dev", ctypes.c_void_p),
        ("expert_events", ctypes.c_void_p),
    ]


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the shared library (once) and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mxfp4_moe_expert_gb300.build`")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.moe_mxfp4_create.argtypes = [ctypes.POINTER(moe_mxfp4_config), ctypes.POINTER(moe_mxfp4_layer),
                                     ctypes.POINTER(P)]
    lib.moe_mxfp4_create.restype = ctypes.c_int
    lib.moe_mxfp4_workspace_bytes.argtypes = [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_mxfp4_workspace_bytes.restype = ctypes.c_int
    lib.moe_mxfp4_forward.argtypes = [P, P, ctypes.c_int32, P, P, ctypes.c_size_t, P,
                                      ctypes.POINTER(moe_mxfp4_debug)]
    lib.moe_mxfp4_forward.restype = ctypes.c_int
    lib.moe_mxfp4_forward_host.argtypes = [P, P, ctypes.c_int32, P, P, ctypes.c_size_t, P]
    lib.moe_mxfp4_forward_host.restype = ctypes.c_int
    lib.moe_mxfp4_check.argtypes = [P, P, P]
    lib.moe_mxfp4_check.restype = ctypes.c_int
    lib.moe_mxfp4_destroy.argtypes = [P]
    lib.moe_mxfp4_destroy.restype = None
    lib.moe_mxfp4_status_string.argtypes = [ctypes.c_int]
    lib.moe_mxfp4_status_string.restype = ctypes.c_char_p
    lib.moe_mxfp4_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P, P]
    lib.moe_mxfp4_quantize.restype = ctypes.c_int
    lib.moe_mxfp4_forward_static.argtypes = [P, P, ctypes.c_int32, P, P]
    lib.moe_mxfp4_forward_static.restype = ctypes.c_int
    lib.moe_mxfp4_accept.argtypes = [P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, P, P, P, P]
    lib.moe_mxfp4_accept.restype = ctypes.c_int
    lib.moe_mxfp4_packed_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_mxfp4_packed_bytes.restype = ctypes.c_int
    lib.moe_mxfp4_pack.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(moe_mxfp4_layer),
                                   P, ctypes.c_size_t, P]
    lib.moe_mxfp4_pack.restype = ctypes.c_int
    lib.moe_mxfp4_split_terms.argtypes = [P, ctypes.c_int64, P, P, P]
    lib.moe_mxfp4_split_terms.restype = ctypes.c_int
    _lib = lib
    return lib


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {moe_mxfp4_status_string(status)} ({status})")


def _check(status: int, what: str) -> int:
    if status != MOE_OK:
        raise MoeError(status, what)
    return status


# ----------------------------------------------------------------------------- C entry points


def moe_mxfp4_status_string(status: int) -> str:
    return load_library().moe_mxfp4_status_string(int(status)).decode()


def moe_mxfp4_create(cfg: moe_mxfp4_config, layers) -> tuple[int, int]:
    """Returns (status, handle).  layers: a sequence of moe_mxfp4_layer."""
    arr = (moe_mxfp4_layer * len(layers))(*layers)
    out = ctypes.c_void_p()
    st = load_library().moe_mxfp4_create(ctypes.byref(cfg), arr, ctypes.byref(out))
    return st, out.value


def moe_mxfp4_workspace_bytes(handle: int, num_tokens: int) -> tuple[int, int]:
    n = ctypes.c_size_t()
    st = load_library().moe_mxfp4_workspace_bytes(handle, num_tokens, ctypes.byref(n))
    return st, n.value


def moe_mxfp4_forward(handle, x_ptr, num_tokens, y_ptr, ws_ptr, ws_bytes, stream_ptr, dbg=None) -> int:
    return load_library().moe_mxfp4_forward(handle, x_ptr, num_tokens, y_ptr, ws_ptr, ws_bytes, stream_ptr,
                                            ctypes.byref(dbg) if dbg is not None else None)


def moe_mxfp4_forward_host(handle, x_host_ptr, num_tokens, y_host_ptr, ws_ptr, ws_bytes, stream_ptr) -> int:
    return load_library().moe_mxfp4_forward_host(handle, x_host_ptr, num_tokens, y_host_ptr, ws_ptr, ws_bytes,
                                                 stream_ptr)


def moe_mxfp4_check(handle, ws_ptr, stream_ptr) -> int:
    return load_library().moe_mxfp4_check(handle, ws_ptr, stream_ptr)


def moe_mxfp4_destroy(handle) -> None:
    if handle:
        load_library().moe_mxfp4_destroy(handle)


def moe_mxfp4_quantize(w_ptr, rows, cols, q_ptr, s_ptr, stream_ptr) -> int:
    return load_library().moe_mxfp4_quantize(w_ptr, rows, cols, q_ptr, s_ptr, stream_ptr)


def moe_mxfp4_forward_static(handle, x_ptr, num_tokens, y_ptr, stream_ptr) -> int:
    """Forward with the library's own static workspace (no device allocation
    anywhere); synchronises the stream and returns the device status."""
    return load_library().moe_mxfp4_forward_static(handle, x_ptr, num_tokens, y_ptr, stream_ptr)


def moe_mxfp4_packed_bytes(hidden, inter, num_experts) -> tuple[int, int]:
    n = ctypes.c_size_t()
    st = load_library().moe_mxfp4_packed_bytes(hidden, inter, num_experts, ctypes.byref(n))
    return st, n.value


def moe_mxfp4_pack(hidden, inter, num_experts, layer: moe_mxfp4_layer, packed_ptr, packed_bytes, stream_ptr) -> int:
    return load_library().moe_mxfp4_pack(hidden, inter, num_experts, ctypes.byref(layer), packed_ptr, packed_bytes,
                                         stream_ptr)


def moe_mxfp4_split_terms(x_ptr, n_blocks, codes_ptr, scales_ptr, stream_ptr) -> int:
    return load_library().moe_mxfp4_split_terms(x_ptr, n_blocks, codes_ptr, scales_ptr, stream_ptr)


# ----------------------------------------------------------------------------- torch convenience


def _layer_desc(L) -> moe_mxfp4_layer:
    def p(name):
        t = L.get(name)
        return t.data_ptr() if t is not None else None
    return moe_mxfp4_layer(p("router_w"), p("router_b"), p("gate_q"), p("gate_s"), p("up_q"), p("up_s"),
                           p("down_q"), p("down_s"), p("norm_w"), p("packed"))


def pack(layer: dict, hidden: int, inter: int, num_experts: int, stream=None):
    """The packed (tile-major) copy of one layer's experts (moe_mxfp4_pack) as a new uint8
    CUDA tensor; `layer` holds the canonical gate_q .. down_s tensors."""
    import torch
    dev = layer["gate_q"].device
    st_, n = moe_mxfp4_packed_bytes(hidden, inter, num_experts)
    _check(st_, "moe_mxfp4_packed_bytes")
    out = torch.empty(n + 256, dtype=torch.uint8, device=dev)
    off = (-out.data_ptr()) % 256                     # 256-byte aligned view
    out = out[off:off + n]
    st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
    canon = {k: v for k, v in layer.items() if k != "packed"}
    _check(moe_mxfp4_pack(hidden, inter, num_experts, _layer_desc(canon), out.data_ptr(), n, st), "moe_mxfp4_pack")
    return out


def moe_mxfp4_accept(logits_ptr, tokens_ptr, num_streams, block, vocab, target_ptr, accepted_ptr,
                     next_token_ptr, stream_ptr) -> int:
    return load_library().moe_mxfp4_accept(logits_ptr, tokens_ptr, num_streams, block, vocab, target_ptr,
                                           accepted_ptr, next_token_ptr, stream_ptr)


def accept(logits, tokens, stream=None):
    """logits: fp32 CUDA [S, B, V]; tokens: int32 CUDA [S, B].  Returns (target [S, B],
    accepted [S], next_token [S]) as int32 CUDA tensors (see moe_mxfp4_accept)."""
    import torch
    S, B, V = logits.shape
    target = torch.empty((S, B), dtype=torch.int32, device=logits.device)
    acc = torch.empty((S,), dtype=torch.int32, device=logits.device)
    nxt = torch.empty((S,), dtype=torch.int32, device=logits.device)
    st = stream if stream is not None else torch.cuda.current_stream(logits.device).cuda_stream
    _check(moe_mxfp4_accept(logits.data_ptr(), tokens.data_ptr(), S, B, V, target.data_ptr(), acc.data_ptr(),
                            nxt.data_ptr(), st), "moe_mxfp4_accept")
    return target, acc, nxt


def split_terms(x, stream=None):
    """x: fp32 CUDA [n, 32] blocks.  Returns (codes uint32 [n, 32], scales uint8 [n, 8])."""
    import torch
    n = x.shape[0]
    codes = torch.empty((n, 32), dtype=torch.int32, device=x.device)
    scales = torch.empty((n, 8), dtype=torch.uint8, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
    _check(moe_mxfp4_split_terms(x.data_ptr(), n, codes.data_ptr(), scales.data_ptr(), st), "moe_mxfp4_split_terms")
    return codes, scales


def quantize(w, q=None, s=None, stream=None):
    """MXFP4-encodes an fp32 CUDA tensor [rows, cols] with the library kernel."""
    import torch
    assert w.is_cuda and w.dtype == torch.float32 and w.dim() == 2 and w.is_contiguous()
    rows, cols = w.shape
    q = q if q is not None else torch.empty((rows, cols // 2), dtype=torch.uint8, device=w.device)
    s = s if s is not None else torch.empty((rows, cols // 32), dtype=torch.uint8, device=w.device)
    st = stream if stream is not None else torch.cuda.current_stream(w.device).cuda_stream
    _check(moe_mxfp4_quantize(w.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(), st), "moe_mxfp4_quantize")
    return q, s


class MoeLayers:
    """Owns a handle over caller-provided device tensors (kept alive here).

    layers: list of dicts with router_w (bf16 [E,H]), router_b (fp32 [E] or None),
    gate_q/gate_s/up_q/up_s/down_q/down_s (uint8), norm_w (bf16 [H] or None) and
    optionally packed (the layer's experts in the packed layout, see pack()).
    """

    def __init__(self, *, hidden, inter, num_experts, top_k, max_tokens, layers, flags=0, rms_eps=1e-6,
                 expert_begin=0, expert_end=0, timeout_us=0):
        self._keep = layers
        self.cfg = moe_mxfp4_config(len(layers), hidden, inter, num_experts, top_k, max_tokens, rms_eps, flags,
                                    expert_begin, expert_end, timeout_us)
        descs = [_layer_desc(L) for L in layers]
        self.handle = None
        st, h = moe_mxfp4_create(self.cfg, descs)
        _check(st, "moe_mxfp4_create")
        self.handle = h
        self.hidden, self.top_k, self.num_experts = hidden, top_k, num_experts
        self.num_layers = len(layers)
        self.out_bf16 = bool(flags & MOE_FLAG_OUT_BF16)

    def workspace_bytes(self, num_tokens: int) -> int:
        st, n = moe_mxfp4_workspace_bytes(self.handle, num_tokens)
        _check(st, "moe_mxfp4_workspace_bytes")
        return n

    def new_workspace(self, num_tokens: int, device="cuda"):
        import torch
        return torch.empty(self.workspace_bytes(num_tokens), dtype=torch.uint8, device=device)

    def _own_workspace(self, num_tokens: int, device):
        """The workspace forward() uses when the caller passes none: one per device, kept
        here and grown when a larger block needs more (a workspace carries the persistent
        forward's state section from one forward to the next, so it is not re-allocated)."""
        cache = self.__dict__.setdefault("_ws", {})
        key = str(device)
        need = self.workspace_bytes(num_tokens)
        ws = cache.get(key)
        if ws is None or ws.numel() < need:
            ws = cache[key] = self.new_workspace(num_tokens, device)
        return ws

    def debug_buffers(self, num_tokens: int, device="cuda"):
        import torch
        L, T, k, E = self.num_layers, num_tokens, self.top_k, self.num_experts
        i32 = dict(dtype=torch.int32, device=device)
        bufs = dict(topk_idx=torch.full((L, T, k), -1, **i32),
                    topk_gate=torch.zeros((L, T, k), dtype=torch.float32, device=device),
                    expert_counts=torch.zeros((L, E), **i32), expert_offsets=torch.zeros((L, E + 1), **i32),
                    perm=torch.full((L, T * k), -1, **i32))
        dbg = moe_mxfp4_debug(*(bufs[n].data_ptr() for n in
                                ("topk_idx", "topk_gate", "expert_counts", "expert_offsets", "perm")), None)
        return bufs, dbg

    def expert_timing(self, events):
        """A debug descriptor that only records `events` (2 per layer, torch.cuda.Event
        created with enable_timing) around each layer's expert kernel."""
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        dbg = moe_mxfp4_debug(None, None, None, None, None, ctypes.cast(arr, ctypes.c_void_p))
        dbg._events_keepalive = arr
        return dbg

    def forward(self, x, y=None, workspace=None, stream=None, dbg=None, check=False):
        """x: bf16 CUDA [T, H].  Returns y (fp32, or bf16 with MOE_FLAG_OUT_BF16)."""
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.hidden), dtype=torch.bfloat16 if self.out_bf16 else torch.float32,
                            device=x.device)
        if workspace is None:
            workspace = self._own_workspace(T, x.device)
        st = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        _check(moe_mxfp4_forward(self.handle, x.data_ptr(), T, y.data_ptr(), workspace.data_ptr(),
                                 workspace.numel(), st, dbg), "moe_mxfp4_forward")
        if check:
            _check(moe_mxfp4_check(self.handle, workspace.data_ptr(), st), "moe_mxfp4_check")
        return y

    def forward_host(self, x_host, y_host, workspace, stream=None):
        import torch
        st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        return _check(moe_mxfp4_forward_host(self.handle, x_host.data_ptr(), x_host.shape[0], y_host.data_ptr(),
                                             workspace.data_ptr(), workspace.numel(), st), "moe_mxfp4_forward_host")

    def close(self):
        if getattr(self, "handle", None):
            moe_mxfp4_destroy(self.handle)
            self.handle = None
        self.__dict__.pop("_ws", None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
