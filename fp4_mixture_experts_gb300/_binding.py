"""ctypes binding of libmoe_fp4.so: argument marshalling only.

Each function mirrors one C entry point of include/moe_fp4.h and takes torch
tensors (device tensors unless stated), passing their data pointers and the
current CUDA stream.  A nonzero status becomes a MoeFp4Error.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmoe_fp4.so"

FLAG_FORCE_GEMV = 0x1
FLAG_FORCE_TC = 0x2
FLAG_PERSISTENT = 0x4
FLAG_CTA_PAIRS = 0x8
FLAG_DETERMINISTIC = 0x10

FAULT_NONE = 0
FAULT_TC_TOKEN_TILE = 1
FAULT_STREAM_STAGE = 2

EXPORTED_SYMBOLS = (
    "moe_fp4_workspace_bytes",
    "moe_fp4_host_workspace_bytes",
    "moe_fp4_route",
    "moe_fp4_router",
    "moe_fp4_forward_gated",
    "moe_fp4_forward",
    "moe_fp4_forward_profiled",
    "moe_fp4_forward_host",
    "moe_fp4_forward_noalloc",
    "moe_fp4_noalloc_check",
    "moe_fp4_set_fault_injection",
    "moe_fp4_mxfp8_quantize",
    "moe_fp4_mx_workspace_bytes",
    "moe_fp4_forward_mx",
    "moe_fp4_check",
    "moe_fp4_status_string",
)


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


class MoeFp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def lib_path() -> str:
    return os.environ.get("MOE_FP4_LIB", os.path.join(PKG, _LIB_NAME))


def load_library():
    """Load the in-tree library (built by fp4_mixture_experts_gb300.build); raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m fp4_mixture_experts_gb300.build` "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    pd = ctypes.POINTER(Dims)
    lib.moe_fp4_workspace_bytes.argtypes = [pd]
    lib.moe_fp4_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_fp4_host_workspace_bytes.argtypes = [pd]
    lib.moe_fp4_host_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_fp4_route.argtypes = [pd, P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.moe_fp4_route.restype = ctypes.c_int
    lib.moe_fp4_forward.argtypes = [pd, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_uint, P, ctypes.c_size_t, P]
    lib.moe_fp4_forward.restype = ctypes.c_int
    lib.moe_fp4_router.argtypes = [pd, P, P, P, P]
    lib.moe_fp4_router.restype = ctypes.c_int
    lib.moe_fp4_forward_gated.argtypes = [pd, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_uint, P,
                                          ctypes.c_size_t, P]
    lib.moe_fp4_forward_gated.restype = ctypes.c_int
    lib.moe_fp4_forward_profiled.argtypes = lib.moe_fp4_forward.argtypes + [ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_fp4_forward_profiled.restype = ctypes.c_int
    lib.moe_fp4_forward_host.argtypes = [pd, P, P, P, P, P, P, P, ctypes.c_uint, P, ctypes.c_size_t, P]
    lib.moe_fp4_forward_host.restype = ctypes.c_int
    lib.moe_fp4_forward_noalloc.argtypes = [pd, P, P, P, P, P, P, P, ctypes.c_uint, P]
    lib.moe_fp4_forward_noalloc.restype = ctypes.c_int
    lib.moe_fp4_noalloc_check.argtypes = [P]
    lib.moe_fp4_noalloc_check.restype = ctypes.c_int
    lib.moe_fp4_set_fault_injection.argtypes = [ctypes.c_int, ctypes.c_uint32]
    lib.moe_fp4_set_fault_injection.restype = ctypes.c_int
    lib.moe_fp4_mxfp8_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P]
    lib.moe_fp4_mxfp8_quantize.restype = ctypes.c_int
    lib.moe_fp4_mx_workspace_bytes.argtypes = [pd]
    lib.moe_fp4_mx_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_fp4_forward_mx.argtypes = [pd, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P,
                                       ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_fp4_forward_mx.restype = ctypes.c_int
    lib.moe_fp4_check.argtypes = [P, P]
    lib.moe_fp4_check.restype = ctypes.c_int
    lib.moe_fp4_status_string.argtypes = [ctypes.c_int]
    lib.moe_fp4_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().moe_fp4_status_string(int(status)).decode()


def _dims(T, d, I, E, k) -> Dims:
    return Dims(int(T), int(d), int(I), int(E), int(k))


def workspace_bytes(T, d, I, E, k) -> int:
    return int(load_library().moe_fp4_workspace_bytes(ctypes.byref(_dims(T, d, I, E, k))))


def host_workspace_bytes(T, d, I, E, k) -> int:
    return int(load_library().moe_fp4_host_workspace_bytes(ctypes.byref(_dims(T, d, I, E, k))))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _events(stage_events):
    """ctypes array of cudaEvent_t handles (torch.cuda.Event, each recorded once so that it exists), or None"""
    if stage_events is None:
        return None
    if len(stage_events) != 6:
        raise ValueError("stage_events takes 6 events")
    return (ctypes.c_void_p * len(stage_events))(*[ctypes.c_void_p(ev.cuda_event) for ev in stage_events])


def _workspace(nbytes, device, workspace):
    import torch
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace has {workspace.numel()} bytes, needs {nbytes}")
    return workspace


def route(router_logits, k: int, d: int = 128, I: int = 128, workspace=None, stream=None):
    """Top-k routing and the expert sort.  router_logits: fp32 [T, E] on the GPU.

    Returns (topk_ids int32 [T, k], topk_weights fp32 [T, k], expert_offsets int32 [E+1],
    sorted_slot int32 [T*k]).  d and I only size the workspace (the routing part does not use them).
    """
    import torch
    T, E = router_logits.shape
    dims = _dims(T, d, I, E, k)
    lib = load_library()
    nbytes = lib.moe_fp4_workspace_bytes(ctypes.byref(dims))
    if nbytes == 0:
        raise MoeFp4Error(-2, "moe_fp4_route")
    dev = router_logits.device
    ws = _workspace(nbytes, dev, workspace)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ss = torch.empty(T * k, dtype=torch.int32, device=dev)
    rc = lib.moe_fp4_route(ctypes.byref(dims), _ptr(router_logits), _ptr(ids), _ptr(w), _ptr(off), _ptr(ss),
                           _ptr(ws), ws.numel(), _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_route")
    return ids, w, off, ss


def mxfp8_quantize(x_bf16, codes=None, scales=None, stream=None):
    """MXFP8 of bf16 rows x_bf16 [R, K] (K a multiple of 32) on the GPU.

    Returns (codes uint8 [R, K] E4M3, scales uint8 [R, K/32] E8M0)."""
    import torch
    if x_bf16.dim() != 2 or x_bf16.dtype != torch.bfloat16 or not x_bf16.is_contiguous():
        raise ValueError("x_bf16 must be a contiguous bf16 [R, K] tensor")
    R, K = x_bf16.shape
    dev = x_bf16.device
    if codes is None:
        codes = torch.empty(R, K, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(R, K // 32, dtype=torch.uint8, device=dev)
    rc = load_library().moe_fp4_mxfp8_quantize(_ptr(x_bf16), R, K, _ptr(codes), _ptr(scales), _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_mxfp8_quantize")
    return codes, scales


def forward(x_bf16, router_logits, w13, w13_scale, w2, w2_scale, k: int, out=None, flags: int = 0,
            workspace=None, return_routing: bool = False, return_h: bool = False, stream=None,
            stage_events=None):
    """The whole layer on device tensors.

    x_bf16: bf16 [T, d]; router_logits: fp32 [T, E]; w13: uint8 [E, 2I, d/2];
    w13_scale: uint8 [E, 2I, d/32]; w2: uint8 [E, d, I/2]; w2_scale: uint8 [E, d, I/32].
    Returns out fp32 [T, d], or a dict with out and the requested extras.
    """
    import torch
    T, d = x_bf16.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dims = _dims(T, d, I, E, k)
    lib = load_library()
    nbytes = lib.moe_fp4_workspace_bytes(ctypes.byref(dims))
    if nbytes == 0:
        raise MoeFp4Error(-2, "moe_fp4_forward")
    dev = x_bf16.device
    ws = _workspace(nbytes, dev, workspace)
    if out is None:
        out = torch.empty(T, d, dtype=torch.float32, device=dev)
    extras = {}
    if return_routing:
        extras = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
                      topk_weights=torch.empty(T, k, dtype=torch.float32, device=dev),
                      expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                      sorted_slot=torch.empty(T * k, dtype=torch.int32, device=dev))
    if return_h:
        extras["h"] = torch.empty(T * k, I, dtype=torch.bfloat16, device=dev)
    args = [ctypes.byref(dims), _ptr(x_bf16), _ptr(router_logits), _ptr(w13), _ptr(w13_scale),
            _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(extras.get("topk_ids")),
            _ptr(extras.get("topk_weights")), _ptr(extras.get("expert_offsets")),
            _ptr(extras.get("sorted_slot")), _ptr(extras.get("h")), int(flags), _ptr(ws),
            ws.numel(), _stream(stream)]
    if stage_events is not None:
        rc = lib.moe_fp4_forward_profiled(*args, _events(stage_events))
    else:
        rc = lib.moe_fp4_forward(*args)
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_forward")
    if extras:
        extras["out"] = out
        return extras
    return out


def mx_workspace_bytes(T, d, I, E, k) -> int:
    return int(load_library().moe_fp4_mx_workspace_bytes(ctypes.byref(_dims(T, d, I, E, k))))


def forward_mx(x_bf16, router_logits, w13, w13_scale, w2, w2_scale, k: int, out=None, workspace=None,
               return_operands: bool = False, stream=None, stage_events=None):
    """The layer with MXFP8 activations on block-scaled tensor cores
    (moe_fp4_forward_mx).  Arguments as in forward; w13 and w2 32-byte aligned.
    Returns out fp32 [T, d], or with return_operands a dict with out and, in
    sorted-row order, h (bf16 [S, I]), h_codes / h_scales (MXFP8 of h) and
    x_codes / x_scales (MXFP8 of each row's token)."""
    import torch
    T, d = x_bf16.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dims = _dims(T, d, I, E, k)
    lib = load_library()
    nbytes = lib.moe_fp4_mx_workspace_bytes(ctypes.byref(dims))
    if nbytes == 0:
        raise MoeFp4Error(-2, "moe_fp4_forward_mx")
    dev = x_bf16.device
    ws = _workspace(nbytes, dev, workspace)
    if out is None:
        out = torch.empty(T, d, dtype=torch.float32, device=dev)
    S = T * k
    ex = {}
    if return_operands:
        ex = dict(h=torch.empty(S, I, dtype=torch.bfloat16, device=dev),
                  h_codes=torch.empty(S, I, dtype=torch.uint8, device=dev),
                  h_scales=torch.empty(S, I // 32, dtype=torch.uint8, device=dev),
                  x_codes=torch.empty(S, d, dtype=torch.uint8, device=dev),
                  x_scales=torch.empty(S, d // 32, dtype=torch.uint8, device=dev))
    rc = lib.moe_fp4_forward_mx(ctypes.byref(dims), _ptr(x_bf16), _ptr(router_logits), _ptr(w13), _ptr(w13_scale),
                                _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(ex.get("h")), _ptr(ex.get("h_codes")),
                                _ptr(ex.get("h_scales")), _ptr(ex.get("x_codes")), _ptr(ex.get("x_scales")),
                                _ptr(ws), ws.numel(), _stream(stream), _events(stage_events))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_forward_mx")
    if ex:
        ex["out"] = out
        return ex
    return out


def router(x_bf16, w_gate_bf16, logits=None, stream=None):
    """Router logits fp32 [T, E] = x (bf16 [T, d]) . w_gate (bf16 [E, d])^T on the GPU."""
    import torch
    T, d = x_bf16.shape
    E = w_gate_bf16.shape[0]
    if w_gate_bf16.shape[1] != d:
        raise ValueError("w_gate must be [E, d]")
    dims = _dims(T, d, 128, E, 1)
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=x_bf16.device)
    rc = load_library().moe_fp4_router(ctypes.byref(dims), _ptr(x_bf16), _ptr(w_gate_bf16), _ptr(logits),
                                       _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_router")
    return logits


def forward_gated(x_bf16, w_gate_bf16, w13, w13_scale, w2, w2_scale, k: int, out=None, flags: int = 0,
                  workspace=None, return_routing: bool = False, return_h: bool = False, stream=None):
    """The whole layer from x and the router weights (bf16 [E, d]).  Returns a
    dict with out and router_logits, plus the requested extras."""
    import torch
    T, d = x_bf16.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dims = _dims(T, d, I, E, k)
    lib = load_library()
    nbytes = lib.moe_fp4_workspace_bytes(ctypes.byref(dims))
    if nbytes == 0:
        raise MoeFp4Error(-2, "moe_fp4_forward_gated")
    dev = x_bf16.device
    ws = _workspace(nbytes, dev, workspace)
    if out is None:
        out = torch.empty(T, d, dtype=torch.float32, device=dev)
    res = {"out": out, "router_logits": torch.empty(T, E, dtype=torch.float32, device=dev)}
    if return_routing:
        res.update(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
                   topk_weights=torch.empty(T, k, dtype=torch.float32, device=dev),
                   expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   sorted_slot=torch.empty(T * k, dtype=torch.int32, device=dev))
    if return_h:
        res["h"] = torch.empty(T * k, I, dtype=torch.bfloat16, device=dev)
    rc = lib.moe_fp4_forward_gated(ctypes.byref(dims), _ptr(x_bf16), _ptr(w_gate_bf16), _ptr(res["router_logits"]),
                                   _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(out),
                                   _ptr(res.get("topk_ids")), _ptr(res.get("topk_weights")),
                                   _ptr(res.get("expert_offsets")), _ptr(res.get("sorted_slot")), _ptr(res.get("h")),
                                   int(flags), _ptr(ws), ws.numel(), _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_forward_gated")
    return res


def forward_host(x_bf16_host, router_logits_host, w13, w13_scale, w2, w2_scale, k: int, out_host=None,
                 flags: int = 0, workspace=None, stream=None):
    """The whole layer with HOST x (bf16 [T, d]), router_logits (fp32 [T, E]) and out (fp32 [T, d]);
    the weights are device tensors.  Synchronises before returning."""
    import torch
    T, d = x_bf16_host.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dims = _dims(T, d, I, E, k)
    lib = load_library()
    nbytes = lib.moe_fp4_host_workspace_bytes(ctypes.byref(dims))
    if nbytes == 0:
        raise MoeFp4Error(-2, "moe_fp4_forward_host")
    ws = _workspace(nbytes, w13.device, workspace)
    if out_host is None:
        out_host = torch.empty(T, d, dtype=torch.float32, pin_memory=x_bf16_host.is_pinned())
    rc = lib.moe_fp4_forward_host(ctypes.byref(dims), _ptr(x_bf16_host), _ptr(router_logits_host), _ptr(w13),
                                  _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(out_host), int(flags), _ptr(ws),
                                  ws.numel(), _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_forward_host")
    return out_host


def forward_noalloc(x_bf16, router_logits, w13, w13_scale, w2, w2_scale, k: int, out=None, flags: int = 0,
                    stream=None):
    """The whole layer with no workspace argument: the library's own fixed
    device scratch is used (see moe_fp4_forward_noalloc in include/moe_fp4.h:
    calls share it, so order them on one stream)."""
    import torch
    T, d = x_bf16.shape
    E, twoI, _ = w13.shape
    dims = _dims(T, d, twoI // 2, E, k)
    if out is None:
        out = torch.empty(T, d, dtype=torch.float32, device=x_bf16.device)
    rc = load_library().moe_fp4_forward_noalloc(ctypes.byref(dims), _ptr(x_bf16), _ptr(router_logits), _ptr(w13),
                                                _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(out), int(flags),
                                                _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_forward_noalloc")
    return out


def check(workspace, stream=None) -> None:
    """Synchronise and raise if a kernel of an earlier call on this workspace
    reported an error (bit 1: an out-of-range expert index; bit 2: a pipeline
    wait that ran out); the error word is cleared."""
    rc = load_library().moe_fp4_check(_ptr(workspace), _stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_check")


def noalloc_check(stream=None) -> None:
    """check() for the internal scratch of forward_noalloc."""
    rc = load_library().moe_fp4_noalloc_check(_stream(stream))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_noalloc_check")


def set_fault_injection(site: int, wait_limit_us: int = 0) -> None:
    """Plant a host-chosen fault in later forward calls (failure-path tests
    only; see moe_fp4_set_fault_injection).  FAULT_NONE restores normal runs."""
    rc = load_library().moe_fp4_set_fault_injection(int(site), int(wait_limit_us))
    if rc != 0:
        raise MoeFp4Error(rc, "moe_fp4_set_fault_injection")
