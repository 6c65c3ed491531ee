"""Thin ctypes binding of the C ABI in include/moe.h.

Argument marshalling only: torch tensors supply device pointers (``data_ptr()``) and the
current CUDA stream; every step of the layer runs in the library's CUDA kernels.  The
functions carry the C names.  A missing or unbuildable library raises -- there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MOE_OK = 0
MOE_ERR_DEVICE_TIMEOUT = -6

_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({moe_error_string(status)})")
        self.status = status


class MoeShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "K", "I", "I_shared")]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W_gate", "bias", "W1", "W3", "W2", "W1s",
                                               "W3s", "W2s")]


class MoeWorkspaceLayout(ctypes.Structure):
    """moe_workspace_layout_t: byte offsets of the layer's intermediates in the workspace."""
    _fields_ = [(n, ctypes.c_size_t) for n in ("offsets", "perm", "slot_pos", "Xp", "h", "Yp",
                                               "Ysh", "bytes")]


class MoeRouting(ctypes.Structure):
    """moe_routing_t: scoring (0 sigmoid, 1 softmax), n_group, topk_group, group_top,
    renorm.  The defaults are the plain router."""
    _fields_ = [(n, ctypes.c_int32) for n in ("scoring", "n_group", "topk_group",
                                              "group_top", "renorm")]

    @classmethod
    def make(cls, scoring: str = "sigmoid", n_group: int = 1, topk_group: int = 1,
             group_top: int = 1, renorm: bool = True) -> "MoeRouting":
        return cls({"sigmoid": 0, "softmax": 1}[scoring], int(n_group), int(topk_group),
                   int(group_top), int(bool(renorm)))


class MoeWeightsFp8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W_gate", "bias", "W1", "W3", "W2", "S1", "S3",
                                               "S2", "W1s", "W3s", "W2s", "S1s", "S3s", "S2s")]


class MoeGraceReplication(ctypes.Structure):
    _fields_ = [("heaviest", ctypes.c_int32), ("n_replica", ctypes.c_int32),
                ("n_hot", ctypes.c_int32), ("rho", ctypes.c_double), ("W_mean", ctypes.c_double),
                ("W_max", ctypes.c_longlong), ("W_r", ctypes.c_longlong)]


def _routing(routing):
    if routing is None:
        return None
    if isinstance(routing, dict):
        routing = MoeRouting.make(**routing)
    return ctypes.byref(routing)


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmoe_gb300.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; run the package build first")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_workspace_bytes": ([ctypes.POINTER(MoeShape)], Z),
        "moe_workspace_layout": ([ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWorkspaceLayout)], I),
        "moe_error_string": ([I], ctypes.c_char_p),
        "moe_read_status": ([P, P], I),
        "moe_debug_set_wait_limit": ([ctypes.c_ulonglong, I], None),
        "moe_debug_set_stage_events": ([P, I], None),
        "moe_debug_set_ffn_variant": ([I], None),
        "moe_debug_set_shared_side": ([I], None),
        "moe_debug_set_sync_status": ([I], None),
        "moe_router_topk": ([P, P, P, I, I, I, I, P, P, P, Z, P], I),
        "moe_router_topk_ex": ([P, P, P, I, I, I, I, ctypes.POINTER(MoeRouting), P, P, P, Z,
                                P], I),
        "moe_router_topk_noalloc": ([P, P, P, I, I, I, I, P, P, P], I),
        "moe_router_topk_noalloc_status": ([P], I),
        "moe_dispatch": ([P, P, I, I, I, I, P, P, P, P, P, P, P, Z, P], I),
        "moe_expert_ffn": ([P, P, I, I, I, I, P, P, P, P, I, P, Z, P], I),
        "moe_expert_ffn_workspace_bytes": ([I, I, I], Z),
        "moe_combine": ([P, P, P, P, I, I, I, P, P], I),
        "moe_layer_forward": ([ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeights), P, P, P,
                               P, P, P, P, Z, P], I),
        "moe_layer_forward_ex": ([ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeights),
                                  ctypes.POINTER(MoeRouting), P, P, P, P, P, P, P, Z, P], I),
        "moe_quantize_weight_fp8": ([P, I, I, I, P, P, P], I),
        "moe_quantize_rows_fp8": ([P, ctypes.c_longlong, I, P, P], I),
        "moe_layer_forward_fp8": ([ctypes.POINTER(MoeShape), ctypes.POINTER(MoeWeightsFp8),
                                   ctypes.POINTER(MoeRouting), P, P, P, P, P, P, P, Z, P], I),
        "moe_grace_metrics": ([P, I, P, I, P, P], I),
        "moe_grace_group": ([P, I, I, ctypes.c_double, P], I),
        "moe_grace_choose_r": ([P, I, I, P, I, P, P, P, P], I),
        "moe_grace_replicate": ([P, I, P, I, P, P, P, ctypes.POINTER(MoeGraceReplication)], I),
        "moe_grace_route_table": ([P, I, ctypes.POINTER(MoeGraceReplication), P, I, P, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


BF16, F32, I32, U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def _chk(t, dtype=None, numel=None, name="tensor"):
    """The C ABI takes bare pointers: a tensor of another element type, or smaller than the
    sizes passed beside it, would be misread (or read past its end) by the kernels."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")


def _ptr(t, dtype=None, numel=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (None stays NULL), after _chk."""
    if t is None:
        return None
    _chk(t, dtype, numel, name)
    if not t.is_cuda:
        raise ValueError(f"{name}: device tensors are required")
    if not t.is_contiguous():
        raise ValueError(f"{name}: contiguous tensors are required")
    return ctypes.c_void_p(t.data_ptr())


def _ptrs(*specs):
    """Pointers of (tensor, dtype, numel, name) arguments: every element type and size is
    checked before any device check."""
    for spec in specs:
        _chk(*spec)
    return [_ptr(*spec) for spec in specs]


def _wstruct(cls, weights: dict, specs, io_specs):
    """A weights structure from (name, dtype, numel) specs (a missing name stays NULL), with
    the layer's input / output tensors (io_specs): every type and size is checked first."""
    ws = [(weights.get(n), dt, k, n) for n, dt, k in specs]
    for spec in ws + list(io_specs):
        _chk(*spec)
    return cls(*[None if t is None else _ptr(t, dt, k, n).value for t, dt, k, n in ws])


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


# ------------------------------------------------------------------------- C entry points
def moe_error_string(status: int) -> str:
    return load().moe_error_string(int(status)).decode()


def moe_workspace_bytes(T, H, E, K, I, I_shared) -> int:
    s = MoeShape(T, H, E, K, I, I_shared)
    return int(load().moe_workspace_bytes(ctypes.byref(s)))


def moe_workspace_layout(T, H, E, K, I, I_shared) -> dict:
    """Byte offsets of offsets, perm, slot_pos, Xp, h, Yp and Ysh inside the layer's
    workspace, and its size ("bytes")."""
    s = MoeShape(T, H, E, K, I, I_shared)
    lay = MoeWorkspaceLayout()
    _check("moe_workspace_layout", load().moe_workspace_layout(ctypes.byref(s), ctypes.byref(lay)))
    return {n: int(getattr(lay, n)) for n, _ in MoeWorkspaceLayout._fields_}


def moe_read_status(ws, stream=None) -> int:
    return int(load().moe_read_status(_ptr(ws), _stream(stream)))


def moe_debug_set_wait_limit(limit_ns: int, inject_stall: int = 0) -> None:
    load().moe_debug_set_wait_limit(int(limit_ns), int(inject_stall))


def moe_debug_set_ffn_variant(variant: int) -> None:
    """0: automatic; 1: single-CTA FFN kernel; 2: CTA-pair (2-SM MMA) FFN kernel."""
    load().moe_debug_set_ffn_variant(int(variant))


def moe_debug_set_sync_status(on: bool) -> None:
    """Debug mode: calls synchronise and return their workspace's status word (a device-side
    error then raises MoeError from the call itself)."""
    load().moe_debug_set_sync_status(1 if on else 0)


def moe_debug_set_shared_side(mode: int) -> None:
    """-1: by batch size (default); 0: shared expert in the routed launch; 1: side stream."""
    load().moe_debug_set_shared_side(int(mode))


def moe_debug_set_stage_events(events) -> None:
    """events: list of >= 6 recorded torch.cuda.Event (timing enabled), or None."""
    if events is None:
        load().moe_debug_set_stage_events(None, 0)
        return
    arr = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
    load().moe_debug_set_stage_events(ctypes.cast(arr, ctypes.c_void_p), len(events))


def _router_args(X, W_gate, bias, K, topk_idx, topk_w):
    T, H = X.shape
    E, K = W_gate.shape[0], int(K)
    x, wg, b, i, w = _ptrs((X, BF16, T * H, "X"), (W_gate, BF16, E * H, "W_gate"),
                           (bias, F32, E, "bias"), (topk_idx, I32, T * K, "topk_idx"),
                           (topk_w, F32, T * K, "topk_w"))
    return (x, wg, b, T, H, E, K), (i, w)


def moe_router_topk(X, W_gate, bias, K, topk_idx, topk_w, ws, stream=None):
    a, o = _router_args(X, W_gate, bias, K, topk_idx, topk_w)
    _check("moe_router_topk", load().moe_router_topk(
        *a, *o, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_router_topk_ex(X, W_gate, bias, K, routing, topk_idx, topk_w, ws, stream=None):
    """routing: MoeRouting, a dict of MoeRouting.make keywords, or None (defaults)."""
    a, o = _router_args(X, W_gate, bias, K, topk_idx, topk_w)
    _check("moe_router_topk_ex", load().moe_router_topk_ex(
        *a, _routing(routing), *o, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_router_topk_noalloc(X, W_gate, bias, K, topk_idx, topk_w, stream=None):
    """The router without a workspace (its scratch is a fixed array of the library)."""
    a, o = _router_args(X, W_gate, bias, K, topk_idx, topk_w)
    _check("moe_router_topk_noalloc", load().moe_router_topk_noalloc(*a, *o, _stream(stream)))


def moe_router_topk_noalloc_status(stream=None) -> int:
    return int(load().moe_router_topk_noalloc_status(_stream(stream)))


def moe_dispatch(X, topk_idx, E, counts, offsets, perm, slot_pos, Xp, affinity, ws,
                 stream=None):
    T, H = X.shape
    K, E = topk_idx.shape[1], int(E)
    x, i, c, o, pm, sp, xp, af = _ptrs(
        (X, BF16, T * H, "X"), (topk_idx, I32, T * K, "topk_idx"), (counts, I32, E, "counts"),
        (offsets, I32, E + 1, "offsets"), (perm, I32, T * K, "perm"),
        (slot_pos, I32, T * K, "slot_pos"), (Xp, BF16, T * K * H, "Xp"),
        (affinity, I32, E * E, "affinity"))
    _check("moe_dispatch", load().moe_dispatch(
        x, i, T, H, E, K, c, o, pm, sp, xp, af, _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_expert_ffn_workspace_bytes(rows: int, n_groups: int, I: int) -> int:
    return int(load().moe_expert_ffn_workspace_bytes(int(rows), int(n_groups), int(I)))


def moe_expert_ffn(Xp, offsets, n_groups, W1, W3, W2, Yp, ws, stream=None):
    rows, H = Xp.shape
    I, G = W1.shape[-1], int(n_groups)
    out_fp32 = 1 if Yp.dtype == torch.float32 else 0
    xp, o, w1, w3, w2, yp = _ptrs(
        (Xp, BF16, rows * H, "Xp"), (offsets, I32, G + 1, "offsets"),
        (W1, BF16, G * H * I, "W1"), (W3, BF16, G * H * I, "W3"), (W2, BF16, G * I * H, "W2"),
        (Yp, F32 if out_fp32 else BF16, rows * H, "Yp"))
    _check("moe_expert_ffn", load().moe_expert_ffn(
        xp, o, G, rows, H, I, w1, w3, w2, yp, out_fp32, _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(Yp, slot_pos, topk_w, Ysh, Y, stream=None):
    T, K = slot_pos.shape
    H = Y.shape[1]
    yp, sp, w, ysh, y = _ptrs((Yp, BF16, T * K * H, "Yp"), (slot_pos, I32, T * K, "slot_pos"),
                              (topk_w, F32, T * K, "topk_w"), (Ysh, F32, T * H, "Ysh"),
                              (Y, F32, T * H, "Y"))
    _check("moe_combine", load().moe_combine(yp, sp, w, ysh, T, H, K, y, _stream(stream)))


def _io_specs(shape: MoeShape, X, Y, topk_idx, topk_w, counts, affinity):
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    return [(X, BF16, T * H, "X"), (Y, F32, T * H, "Y"), (topk_idx, I32, T * K, "topk_idx"),
            (topk_w, F32, T * K, "topk_w"), (counts, I32, E, "counts"),
            (affinity, I32, E * E, "affinity")]


def _layer_args(shape: MoeShape, weights: dict, io):
    H, E, I, Is = shape.H, shape.E, shape.I, shape.I_shared
    w = _wstruct(MoeWeights, weights,
                 (("W_gate", BF16, E * H), ("bias", F32, E), ("W1", BF16, E * H * I),
                  ("W3", BF16, E * H * I), ("W2", BF16, E * I * H), ("W1s", BF16, H * Is),
                  ("W3s", BF16, H * Is), ("W2s", BF16, Is * H)), io)
    return w, _ptrs(*io)


def moe_layer_forward(shape: MoeShape, weights: dict, X, Y, topk_idx, topk_w, counts,
                      affinity, ws, stream=None):
    w, io = _layer_args(shape, weights, _io_specs(shape, X, Y, topk_idx, topk_w, counts, affinity))
    _check("moe_layer_forward", load().moe_layer_forward(
        ctypes.byref(shape), ctypes.byref(w), *io, _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_layer_forward_ex(shape: MoeShape, weights: dict, routing, X, Y, topk_idx, topk_w,
                         counts, affinity, ws, stream=None):
    w, io = _layer_args(shape, weights, _io_specs(shape, X, Y, topk_idx, topk_w, counts, affinity))
    _check("moe_layer_forward_ex", load().moe_layer_forward_ex(
        ctypes.byref(shape), ctypes.byref(w), _routing(routing), *io, _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_quantize_weight_fp8(W, stream=None):
    """W bf16 [G, R, C] or [R, C] (device; R the reduction dimension) -> (E4M3 bytes uint8,
    transposed: [G, C, R] or [C, R]; int32 scale exponents [G, R/128, C/128] or
    [R/128, C/128])."""
    shape = W.shape
    G, R, C = (1,) + tuple(shape) if W.dim() == 2 else tuple(shape)
    Wq = torch.empty(shape[:-2] + (C, R), dtype=torch.uint8, device=W.device)
    S = torch.empty(shape[:-2] + (R // 128, C // 128), dtype=torch.int32, device=W.device)
    _check("moe_quantize_weight_fp8", load().moe_quantize_weight_fp8(
        _ptr(W, BF16, name="W"), G, R, C, _ptr(Wq), _ptr(S), _stream(stream)))
    return Wq, S


def moe_quantize_rows_fp8(x, out=None, stream=None):
    rows, n = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_quantize_rows_fp8", load().moe_quantize_rows_fp8(
        _ptr(x), rows, n, _ptr(out), _stream(stream)))
    return out


def quantize_expert_weights_fp8(weights: dict, stream=None) -> dict:
    """bf16 layer weights (W_gate, bias, W1, W3, W2[, W1s, W3s, W2s]) -> the FP8 layer's
    weights (E4M3 bytes and tile scale exponents); W_gate and bias are kept."""
    out = {"W_gate": weights["W_gate"], "bias": weights["bias"]}
    for w, sc in (("W1", "S1"), ("W3", "S3"), ("W2", "S2"), ("W1s", "S1s"), ("W3s", "S3s"),
                  ("W2s", "S2s")):
        if weights.get(w) is None:
            out[w] = out[sc] = None
            continue
        out[w], out[sc] = moe_quantize_weight_fp8(weights[w], stream)
    return out


def moe_layer_forward_fp8(shape: MoeShape, weights8: dict, routing, X, Y, topk_idx, topk_w,
                          counts, affinity, ws, stream=None):
    H, E, I, Is = shape.H, shape.E, shape.I, shape.I_shared
    tiles, tiles_s = (H // 128) * (I // 128), (H // 128) * (Is // 128)
    io = _io_specs(shape, X, Y, topk_idx, topk_w, counts, affinity)
    w = _wstruct(MoeWeightsFp8, weights8,
                 (("W_gate", BF16, E * H), ("bias", F32, E), ("W1", U8, E * H * I),
                  ("W3", U8, E * H * I), ("W2", U8, E * I * H), ("S1", I32, E * tiles),
                  ("S3", I32, E * tiles), ("S2", I32, E * tiles), ("W1s", U8, H * Is),
                  ("W3s", U8, H * Is), ("W2s", U8, Is * H), ("S1s", I32, tiles_s),
                  ("S3s", I32, tiles_s), ("S2s", I32, tiles_s)), io)
    _check("moe_layer_forward_fp8", load().moe_layer_forward_fp8(
        ctypes.byref(shape), ctypes.byref(w), _routing(routing), *_ptrs(*io), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


# ------------------------------------------------------------------- convenience wrapper
class MoELayer:
    """Holds a layer's weights, outputs and workspace (torch allocations) and runs
    moe_layer_forward.  weights: dict of device tensors W_gate, bias, W1, W3, W2 and
    (optionally) W1s, W3s, W2s."""

    def __init__(self, weights: dict, T: int, K: int, with_affinity: bool = True,
                 routing=None, fp8: bool = False, weights8: dict | None = None):
        self.w = weights
        self.routing = routing
        # FP8 experts: the weights are quantised once here (static, 128 x 128 tiles), unless
        # another layer's quantised weights are passed in
        self.w8 = (weights8 if weights8 is not None else quantize_expert_weights_fp8(weights)) if fp8 else None
        E, H = weights["W_gate"].shape
        I = weights["W1"].shape[-1]
        Is = 0 if weights.get("W1s") is None else weights["W1s"].shape[-1]
        self.shape = MoeShape(T, H, E, K, I, Is)
        dev = weights["W_gate"].device
        self.Y = torch.empty(T, H, dtype=torch.float32, device=dev)
        self.topk_idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        self.topk_w = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.affinity = (torch.empty(E, E, dtype=torch.int32, device=dev)
                         if with_affinity else None)
        nbytes = moe_workspace_bytes(T, H, E, K, I, Is)
        if nbytes == 0:
            raise MoeError("moe_workspace_bytes", -2)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def forward(self, X, stream=None):
        if self.w8 is not None:
            moe_layer_forward_fp8(self.shape, self.w8, self.routing, X, self.Y, self.topk_idx,
                                  self.topk_w, self.counts, self.affinity, self.ws, stream)
        elif self.routing is None:
            moe_layer_forward(self.shape, self.w, X, self.Y, self.topk_idx, self.topk_w,
                              self.counts, self.affinity, self.ws, stream)
        else:
            moe_layer_forward_ex(self.shape, self.w, self.routing, X, self.Y, self.topk_idx,
                                 self.topk_w, self.counts, self.affinity, self.ws, stream)
        return self.Y

    def status(self, stream=None) -> int:
        return moe_read_status(self.ws, stream)

    def intermediates(self) -> dict:
        """Views (no copies) of the last forward's offsets [E+1], perm [T*K], slot_pos
        [T,K] and Xp [T*K,H] inside the workspace (moe_workspace_layout)."""
        s = self.shape
        lay = moe_workspace_layout(s.T, s.H, s.E, s.K, s.I, s.I_shared)
        TK = s.T * s.K

        def view(off, n, dtype, shape):
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            return self.ws[off:off + nbytes].view(dtype).view(*shape)
        return dict(offsets=view(lay["offsets"], s.E + 1, torch.int32, (s.E + 1,)),
                    perm=view(lay["perm"], TK, torch.int32, (TK,)),
                    slot_pos=view(lay["slot_pos"], TK, torch.int32, (s.T, s.K)),
                    Xp=view(lay["Xp"], TK * s.H, torch.bfloat16, (TK, s.H)))


# ------------------------------------------------------ GRACE-MoE placement (host arrays)
def _np(a, dtype):
    import numpy as np
    return np.ascontiguousarray(a, dtype=dtype)


def _hp(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def moe_grace_metrics(affinity, group_of, D: int):
    import numpy as np
    A = _np(affinity, np.int32)
    g = _np(group_of, np.int32)
    U, S = ctypes.c_double(), ctypes.c_double()
    _check("moe_grace_metrics", load().moe_grace_metrics(_hp(A), A.shape[0], _hp(g), int(D),
                                                         ctypes.byref(U), ctypes.byref(S)))
    return U.value, S.value


def moe_grace_group(affinity, D: int, r: float):
    import numpy as np
    A = _np(affinity, np.int32)
    g = np.zeros(A.shape[0], np.int32)
    _check("moe_grace_group", load().moe_grace_group(_hp(A), A.shape[0], int(D), float(r), _hp(g)))
    return g


def moe_grace_choose_r(affinity, D: int, r_grid):
    import numpy as np
    A = _np(affinity, np.int32)
    r = _np(r_grid, np.float64)
    U, S = np.zeros(len(r)), np.zeros(len(r))
    g = np.zeros(A.shape[0], np.int32)
    k = ctypes.c_int()
    _check("moe_grace_choose_r", load().moe_grace_choose_r(
        _hp(A), A.shape[0], int(D), _hp(r), len(r), _hp(U), _hp(S), ctypes.byref(k), _hp(g)))
    return dict(U=U, S=S, knee=k.value, r=float(r[k.value]), group_of=g)


def moe_grace_replicate(counts, group_of, D: int):
    import numpy as np
    c = _np(counts, np.int32)
    g = _np(group_of, np.int32)
    W = np.zeros(D, np.int64)
    hot = np.zeros(len(c), np.int32)
    rg = np.zeros(max(D - 1, 1), np.int32)
    rep = MoeGraceReplication()
    _check("moe_grace_replicate", load().moe_grace_replicate(
        _hp(c), len(c), _hp(g), int(D), _hp(W), _hp(hot), _hp(rg), ctypes.byref(rep)))
    return dict(W=W.tolist(), W_mean=rep.W_mean, W_max=rep.W_max, heaviest=rep.heaviest,
                rho=rep.rho, n_replica=rep.n_replica, hot=hot[:rep.n_hot].tolist(),
                W_r=rep.W_r, replica_gpus=rg[:rep.n_replica].tolist(), _struct=rep)


def moe_grace_route_table(rep: dict, gpus_per_node: int):
    import numpy as np
    W = _np(rep["W"], np.int64)
    D = len(W)
    st = rep["_struct"]
    rg = _np(rep["replica_gpus"] or [0], np.int32)
    n = 1 + st.n_replica
    pred = np.zeros(n)
    table = np.zeros((D, n))
    _check("moe_grace_route_table", load().moe_grace_route_table(
        _hp(W), D, ctypes.byref(st), _hp(rg), int(gpus_per_node), _hp(pred), _hp(table)))
    return dict(instances=[st.heaviest] + list(rep["replica_gpus"]), predicted=pred, table=table)
