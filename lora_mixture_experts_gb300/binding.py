"""ctypes binding of libmoelora.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (declared in
``include/moelora.h``), takes torch tensors for the device buffers and
passes their data pointers and the current CUDA stream.  All arithmetic
happens in the library's kernels; if the library is missing, ``load()``
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

_LIB = None

MOELORA_OK = 0
STATUS = {
    0: "MOELORA_OK", -1: "MOELORA_ERR_INVALID_ARG", -2: "MOELORA_ERR_UNSUPPORTED",
    -3: "MOELORA_ERR_MISALIGNED", -4: "MOELORA_ERR_WORKSPACE", -5: "MOELORA_ERR_CUDA",
    -6: "MOELORA_ERR_BAD_INDEX", -7: "MOELORA_ERR_TIMEOUT", -8: "MOELORA_ERR_DEVICE_CHECK",
}


class MoeLoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class moelora_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "k", "E", "H", "I", "L", "r")]


class moelora_linear_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "K", "N", "L", "r")]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I32 = ctypes.c_int32
_SIGS = {
    "moelora_workspace_bytes": (_SZ, [ctypes.POINTER(moelora_dims)]),
    "moelora_linear_workspace_bytes": (_SZ, [ctypes.POINTER(moelora_linear_dims)]),
    "moelora_align_workspace_bytes": (_SZ, [ctypes.POINTER(moelora_dims)]),
    "moelora_align_capacity": (_SZ, [ctypes.POINTER(moelora_dims), _I32]),
    "moe_lora_align": (ctypes.c_int, [ctypes.POINTER(moelora_dims), _P, _P, _I32, _P, _P, _P, _P,
                                      _P, _SZ, _P]),
    "moe_lora_align_noalloc": (ctypes.c_int, [ctypes.POINTER(moelora_dims), _P, _P, _I32, _P, _P,
                                              _P, _P, _P]),
    "moe_lora_forward": (ctypes.c_int, [ctypes.POINTER(moelora_dims)] + [_P] * 12 + [_SZ, _P]),
    "moe_lora_route": (ctypes.c_int, [ctypes.POINTER(moelora_dims), _P, _P, _P, _P]),
    "moe_lora_forward_routed": (ctypes.c_int, [ctypes.POINTER(moelora_dims)] + [_P] * 11 + [_SZ, _P]),
    "moe_lora_linear": (ctypes.c_int, [ctypes.POINTER(moelora_linear_dims)] + [_P] * 7 + [_SZ, _P]),
    "moe_lora_merge_adapter": (ctypes.c_int, [ctypes.POINTER(moelora_dims), _I32] + [_P] * 8 + [_P]),
    "moelora_load_tuning": (ctypes.c_int, [ctypes.c_char_p]),
    "moelora_tuning_entries": (_I32, []),
    "moelora_set_timing_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), _I32]),
    "moelora_last_launch_count": (_I32, []),
    "moelora_last_launch_name": (ctypes.c_char_p, [_I32]),
    "moelora_get_error": (ctypes.c_int, [_P, _P]),
    "moelora_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


def library_path() -> str:
    """The library to load: libmoelora.so, or the file MOELORA_LIBRARY names
    (the tests point it at the checked debug build)."""
    return os.environ.get("MOELORA_LIBRARY") or _build.LIB


def load(build_if_missing: bool = True):
    """Load the library (building it first if it is missing and nvcc exists)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        if os.environ.get("MOELORA_LIBRARY"):
            raise FileNotFoundError(f"MOELORA_LIBRARY={path} does not exist")
        if not build_if_missing:
            raise FileNotFoundError(f"{path} is not built; run lora_mixture_experts_gb300.build")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def exported_symbols() -> Sequence[str]:
    return list(_SIGS)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors are required")
    if not t.is_contiguous():
        raise ValueError("contiguous tensors are required")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name: str, dtype, shape=None, optional: bool = False):
    """Argument checks the C ABI cannot make (it sees only pointers and the
    sizes passed in moelora_dims): dtype and shape of every tensor, before
    anything is allocated or launched."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _same_device(*ts, stream=None):
    """The tensors share one device, which is the current CUDA device, and an
    explicit stream belongs to it.  The library launches on the current
    device with the pointers it is given, so tensors of another device would
    fault on the GPU instead of raising here."""
    devs = {t.device for t in ts if t is not None}
    if len(devs) > 1:
        raise ValueError(f"tensors on several devices: {sorted(str(d) for d in devs)}")
    if not devs:
        return
    dev = next(iter(devs))
    if dev.type != "cuda":
        return                      # _ptr reports host tensors
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError(f"tensors on {dev} but the current CUDA device is cuda:{cur} "
                         f"(call under torch.cuda.device({dev.index}))")
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream on {stream.device}, tensors on {dev}")


def _check_layer(x, topk_weights, lora_ids, W_gate_up, W_down, A_gu, B_gu, A_d, B_d, out, ws,
                 topk_ids=None, router_logits=None, k=None, stream=None):
    if x.dim() != 2 or W_gate_up.dim() != 3:
        raise ValueError("x must be [T, H] and W_gate_up [E, 2I, H]")
    T, H = x.shape
    E, two_i, _ = W_gate_up.shape
    I = two_i // 2
    bf = torch.bfloat16
    _need(x, "x", bf)
    _need(W_gate_up, "W_gate_up", bf, (E, 2 * I, H))
    _need(W_down, "W_down", bf, (E, H, I))
    if topk_ids is not None:
        if topk_ids.dim() != 2:
            raise ValueError("topk_ids must be [T, k]")
        k = topk_ids.shape[1]
        _need(topk_ids, "topk_ids", torch.int32, (T, k))
        _need(topk_weights, "topk_weights", torch.float32, (T, k))
    if router_logits is not None:
        _need(router_logits, "router_logits", torch.float32, (T, E))
    _need(lora_ids, "lora_ids", torch.int32, (T,))
    if A_gu is not None:
        if A_gu.dim() != 4:
            raise ValueError("A_gu must be [L, E, r, H]")
        L, r = A_gu.shape[0], A_gu.shape[2]
        _need(A_gu, "A_gu", bf, (L, E, r, H))
        _need(B_gu, "B_gu", bf, (L, E, 2 * I, r))
        _need(A_d, "A_d", bf, (L, E, r, I))
        _need(B_d, "B_d", bf, (L, E, H, r))
    _need(out, "out", bf, (T, H), optional=True)
    _need(ws, "ws", torch.uint8, optional=True)
    _same_device(x, topk_ids, topk_weights, router_logits, lora_ids, W_gate_up, W_down, A_gu, B_gu,
                 A_d, B_d, out, ws, stream=stream)


def _check(st: int, where: str):
    if st != MOELORA_OK:
        raise MoeLoraError(st, where)


def dims_of(x, topk_ids, W_gate_up, W_down, A_gu=None) -> moelora_dims:
    T, H = x.shape
    E, two_i, _ = W_gate_up.shape
    L, r = (A_gu.shape[0], A_gu.shape[2]) if A_gu is not None else (0, 0)
    return moelora_dims(T, topk_ids.shape[1], E, H, two_i // 2, L, r)


def moelora_workspace_bytes(d: moelora_dims) -> int:
    return load().moelora_workspace_bytes(ctypes.byref(d))


def moelora_linear_workspace_bytes(d: moelora_linear_dims) -> int:
    return load().moelora_linear_workspace_bytes(ctypes.byref(d))


def moelora_align_workspace_bytes(d: moelora_dims) -> int:
    return load().moelora_align_workspace_bytes(ctypes.byref(d))


def moelora_align_capacity(d: moelora_dims, block_m: int) -> int:
    return load().moelora_align_capacity(ctypes.byref(d), block_m)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def moe_lora_align(topk_ids, lora_ids, E: int, L: int, block_m: int, ws=None, stream=None):
    """Returns (sorted_ids, blk_expert, seg_off, num_post_pad) device tensors."""
    lib = load()
    T, k = topk_ids.shape
    _need(topk_ids, "topk_ids", torch.int32)
    _need(lora_ids, "lora_ids", torch.int32, (T,))
    _need(ws, "ws", torch.uint8, optional=True)
    _same_device(topk_ids, lora_ids, ws, stream=stream)
    d = moelora_dims(T, k, E, 8, 8, L, 0)
    cap = lib.moelora_align_capacity(ctypes.byref(d), block_m)
    dev = topk_ids.device
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    blk = torch.empty(max(cap // max(block_m, 1), 1), dtype=torch.int32, device=dev)
    seg = torch.empty(E * (L + 1) + 1, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = alloc_workspace(lib.moelora_align_workspace_bytes(ctypes.byref(d)), dev)
    st = lib.moe_lora_align(ctypes.byref(d), _ptr(topk_ids), _ptr(lora_ids), block_m,
                            _ptr(sorted_ids), _ptr(blk), _ptr(seg), _ptr(npp), _ptr(ws),
                            ws.numel(), _stream(stream))
    _check(st, "moe_lora_align")
    return sorted_ids[:cap], blk[:cap // block_m], seg, npp


def moe_lora_align_noalloc(topk_ids, lora_ids, E: int, L: int, block_m: int, stream=None):
    """moe_lora_align for callers that cannot allocate device scratch: the
    library uses its own fixed 4 MiB device array instead of a workspace.
    Returns (sorted_ids, blk_expert, seg_off, num_post_pad); the output
    tensors are allocated here by torch only for the caller's convenience."""
    lib = load()
    T, k = topk_ids.shape
    _need(topk_ids, "topk_ids", torch.int32)
    _need(lora_ids, "lora_ids", torch.int32, (T,))
    _same_device(topk_ids, lora_ids, stream=stream)
    d = moelora_dims(T, k, E, 8, 8, L, 0)
    cap = lib.moelora_align_capacity(ctypes.byref(d), block_m)
    dev = topk_ids.device
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    blk = torch.empty(max(cap // max(block_m, 1), 1), dtype=torch.int32, device=dev)
    seg = torch.empty(E * (L + 1) + 1, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    st = lib.moe_lora_align_noalloc(ctypes.byref(d), _ptr(topk_ids), _ptr(lora_ids), block_m,
                                    _ptr(sorted_ids), _ptr(blk), _ptr(seg), _ptr(npp), _stream(stream))
    _check(st, "moe_lora_align_noalloc")
    return sorted_ids[:cap], blk[:cap // block_m], seg, npp


def moe_lora_forward(x, topk_ids, topk_weights, lora_ids, W_gate_up, W_down,
                     A_gu=None, B_gu=None, A_d=None, B_d=None, out=None, ws=None, stream=None):
    """The fused MoE-LoRA expert layer; returns out[T,H] bf16."""
    lib = load()
    _check_layer(x, topk_weights, lora_ids, W_gate_up, W_down, A_gu, B_gu, A_d, B_d, out, ws,
                 topk_ids=topk_ids, stream=stream)
    d = dims_of(x, topk_ids, W_gate_up, W_down, A_gu)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = alloc_workspace(lib.moelora_workspace_bytes(ctypes.byref(d)), x.device)
    st = lib.moe_lora_forward(ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                              _ptr(lora_ids), _ptr(W_gate_up), _ptr(W_down), _ptr(A_gu),
                              _ptr(B_gu), _ptr(A_d), _ptr(B_d), _ptr(out), _ptr(ws), ws.numel(),
                              _stream(stream))
    _check(st, "moe_lora_forward")
    return out


def moe_lora_route(logits, k: int, ids=None, weights=None, stream=None):
    """Router top-k on device: returns (topk_ids [T,k] int32, topk_weights [T,k] fp32)."""
    lib = load()
    T, E = logits.shape
    _need(logits, "logits", torch.float32)
    _need(ids, "ids", torch.int32, (T, k), optional=True)
    _need(weights, "weights", torch.float32, (T, k), optional=True)
    _same_device(logits, ids, weights, stream=stream)
    d = moelora_dims(T, k, E, 8, 8, 0, 0)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    st = lib.moe_lora_route(ctypes.byref(d), _ptr(logits), _ptr(ids), _ptr(weights), _stream(stream))
    _check(st, "moe_lora_route")
    return ids, weights


def moe_lora_forward_routed(x, router_logits, k: int, lora_ids, W_gate_up, W_down,
                            A_gu=None, B_gu=None, A_d=None, B_d=None, out=None, ws=None,
                            stream=None):
    """The layer with the router fused in (router logits [T,E] fp32, top-k)."""
    lib = load()
    _check_layer(x, None, lora_ids, W_gate_up, W_down, A_gu, B_gu, A_d, B_d, out, ws,
                 router_logits=router_logits, stream=stream)
    T, H = x.shape
    E, two_i, _ = W_gate_up.shape
    L, r = (A_gu.shape[0], A_gu.shape[2]) if A_gu is not None else (0, 0)
    d = moelora_dims(T, k, E, H, two_i // 2, L, r)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = alloc_workspace(lib.moelora_workspace_bytes(ctypes.byref(d)), x.device)
    st = lib.moe_lora_forward_routed(ctypes.byref(d), _ptr(x), _ptr(router_logits), _ptr(lora_ids),
                                     _ptr(W_gate_up), _ptr(W_down), _ptr(A_gu), _ptr(B_gu),
                                     _ptr(A_d), _ptr(B_d), _ptr(out), _ptr(ws), ws.numel(),
                                     _stream(stream))
    _check(st, "moe_lora_forward_routed")
    return out


def moe_lora_linear(x, lora_ids, W, A=None, B=None, out=None, ws=None, stream=None):
    """Dense multi-LoRA linear; returns out[T,N] bf16."""
    lib = load()
    T, K = x.shape
    N = W.shape[0]
    L, r = (A.shape[0], A.shape[1]) if A is not None else (0, 0)
    bf = torch.bfloat16
    _need(x, "x", bf)
    _need(lora_ids, "lora_ids", torch.int32, (T,))
    _need(W, "W", bf, (N, K))
    if A is not None:
        _need(A, "A", bf, (L, r, K))
        _need(B, "B", bf, (L, N, r))
    _need(out, "out", bf, (T, N), optional=True)
    _need(ws, "ws", torch.uint8, optional=True)
    _same_device(x, lora_ids, W, A, B, out, ws, stream=stream)
    d = moelora_linear_dims(T, K, N, L, r)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = alloc_workspace(lib.moelora_linear_workspace_bytes(ctypes.byref(d)), x.device)
    st = lib.moe_lora_linear(ctypes.byref(d), _ptr(x), _ptr(lora_ids), _ptr(W), _ptr(A), _ptr(B),
                             _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_lora_linear")
    return out


def moe_lora_merge_adapter(adapter: int, W_gate_up, W_down, A_gu, B_gu, A_d, B_d,
                           W_gate_up_out=None, W_down_out=None, stream=None):
    """W' = W + B A of one adapter for every expert; returns (W_gate_up', W_down')."""
    lib = load()
    E, two_i, H = W_gate_up.shape
    L, _, r, _ = A_gu.shape
    I = two_i // 2
    bf = torch.bfloat16
    _need(W_gate_up, "W_gate_up", bf, (E, 2 * I, H))
    _need(W_down, "W_down", bf, (E, H, I))
    _need(A_gu, "A_gu", bf, (L, E, r, H))
    _need(B_gu, "B_gu", bf, (L, E, 2 * I, r))
    _need(A_d, "A_d", bf, (L, E, r, I))
    _need(B_d, "B_d", bf, (L, E, H, r))
    _need(W_gate_up_out, "W_gate_up_out", bf, (E, 2 * I, H), optional=True)
    _need(W_down_out, "W_down_out", bf, (E, H, I), optional=True)
    _same_device(W_gate_up, W_down, A_gu, B_gu, A_d, B_d, W_gate_up_out, W_down_out, stream=stream)
    d = moelora_dims(0, 1, E, H, two_i // 2, L, r)
    if W_gate_up_out is None:
        W_gate_up_out = torch.empty_like(W_gate_up)
    if W_down_out is None:
        W_down_out = torch.empty_like(W_down)
    st = lib.moe_lora_merge_adapter(ctypes.byref(d), adapter, _ptr(W_gate_up), _ptr(W_down),
                                    _ptr(A_gu), _ptr(B_gu), _ptr(A_d), _ptr(B_d),
                                    _ptr(W_gate_up_out), _ptr(W_down_out), _stream(stream))
    _check(st, "moe_lora_merge_adapter")
    return W_gate_up_out, W_down_out


def moelora_load_tuning(path) -> None:
    """Load (or with None clear) the tuned launch-choice table."""
    p = None if path is None else os.fsencode(path)
    _check(load().moelora_load_tuning(p), "moelora_load_tuning")


def moelora_tuning_entries() -> int:
    return load().moelora_tuning_entries()


def moelora_get_error(ws, stream=None) -> int:
    _same_device(ws, stream=stream)
    return load().moelora_get_error(_ptr(ws), _stream(stream))


def moelora_set_timing_events(events) -> None:
    """Install (list of torch.cuda.Event) or remove (None) the per-launch timing hook."""
    lib = load()
    if not events:
        _check(lib.moelora_set_timing_events(None, 0), "moelora_set_timing_events")
        return
    for e in events:
        e.record() if e.cuda_event == 0 else None   # make sure the event exists
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib.moelora_set_timing_events(arr, len(events)), "moelora_set_timing_events")


def moelora_last_launches():
    lib = load()
    n = lib.moelora_last_launch_count()
    return [lib.moelora_last_launch_name(i).decode() for i in range(n)]


def moelora_status_string(status: int) -> str:
    return load().moelora_status_string(status).decode()
