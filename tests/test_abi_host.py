"""C-ABI checks that need no GPU: the library loads, exports every entry point
``include/moelora.h`` declares, sizes its workspace on the host, and rejects
bad arguments with status codes before anything is enqueued.  Device
pointers here are fake addresses that the library must never dereference
on these paths."""
import ctypes
import os
import re

import pytest

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.binding import moelora_dims, moelora_linear_dims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moelora.h")

OK, INVALID, UNSUP, MISAL, WS = 0, -1, -2, -3, -4
FAKE = 0x7f0000000000          # 256-byte aligned, never dereferenced


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert "moe_lora_forward" in names and "moe_lora_align" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.exported_symbols())


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert binding.moelora_status_string(s) not in ("", "unknown status")


def _d(T=16, k=4, E=32, H=2880, I=2880, L=8, r=32):
    return moelora_dims(T, k, E, H, I, L, r)


def test_workspace_sizes(lib):
    assert binding.moelora_workspace_bytes(_d()) > 0
    # grows with tokens, never zero for valid sizes
    assert binding.moelora_workspace_bytes(_d(T=4096)) > binding.moelora_workspace_bytes(_d(T=16))
    assert binding.moelora_workspace_bytes(_d(T=0)) > 0
    assert binding.moelora_workspace_bytes(_d(L=0, r=0)) < binding.moelora_workspace_bytes(_d())
    assert binding.moelora_workspace_bytes(_d(k=40)) == 0          # k > E
    assert binding.moelora_workspace_bytes(_d(H=2884)) == 0        # H % 8
    assert binding.moelora_workspace_bytes(_d(r=24)) == 0          # rank not supported
    assert binding.moelora_workspace_bytes(_d(E=1024, L=10, k=4)) > 0   # 11264 bins: the limit
    assert binding.moelora_workspace_bytes(_d(E=1024, L=11, k=4)) == 0  # 12288 bins
    assert binding.moelora_workspace_bytes(_d(E=1025, L=0, r=0, k=4)) == 0
    assert binding.moelora_linear_workspace_bytes(moelora_linear_dims(512, 8192, 28672, 32, 16)) > 0
    assert binding.moelora_align_capacity(_d(), 16) == 16 * 4 + 32 * 15
    assert binding.moelora_align_capacity(_d(), 0) == 0
    assert binding.moelora_align_workspace_bytes(_d()) > 0


def _fwd(lib, d, ptrs=None, ws_bytes=1 << 40, ws=FAKE):
    p = [ctypes.c_void_p(FAKE)] * 11 if ptrs is None else ptrs
    return lib.moe_lora_forward(ctypes.byref(d), *p, ctypes.c_void_p(ws), ws_bytes, None)


def test_forward_argument_errors(lib):
    assert _fwd(lib, _d(T=0)) == OK                         # empty batch: no-op
    assert _fwd(lib, _d(k=0)) == INVALID
    assert _fwd(lib, _d(T=-1)) == INVALID
    assert _fwd(lib, _d(k=33)) == INVALID
    assert _fwd(lib, _d(I=2884)) == UNSUP
    assert _fwd(lib, _d(r=8)) == UNSUP
    assert _fwd(lib, _d(r=40)) == UNSUP
    assert _fwd(lib, _d(r=144)) == UNSUP
    assert _fwd(lib, _d(E=2048, k=2)) == UNSUP
    assert _fwd(lib, _d(E=1024, L=11, k=4)) == UNSUP             # E*(L+1) above 11264
    assert _fwd(lib, _d(T=1 << 28, k=4)) == UNSUP                # T*k reaches 2^30
    p = [ctypes.c_void_p(FAKE)] * 11
    p[0] = None                                              # x
    assert _fwd(lib, _d(), p) == INVALID
    p = [ctypes.c_void_p(FAKE)] * 11
    p[7] = None                                              # B_gu with LoRA on
    assert _fwd(lib, _d(), p) == INVALID
    assert _fwd(lib, _d(L=0, r=0), p) != INVALID             # ...fine without LoRA (fails later: ws)
    p = [ctypes.c_void_p(FAKE)] * 11
    p[4] = ctypes.c_void_p(FAKE + 2)                         # W_gate_up misaligned
    assert _fwd(lib, _d(), p) == MISAL
    assert _fwd(lib, _d(), ws=FAKE + 64) == MISAL            # workspace not 256-aligned
    assert _fwd(lib, _d(), ws=0) == WS
    need = binding.moelora_workspace_bytes(_d())
    assert _fwd(lib, _d(), ws_bytes=need - 1) == WS


def test_linear_and_align_argument_errors(lib):
    d = moelora_linear_dims(8, 8192, 28672, 32, 16)
    P = [ctypes.c_void_p(FAKE)] * 6
    assert lib.moe_lora_linear(ctypes.byref(moelora_linear_dims(0, 8192, 28672, 32, 16)), *P,
                               ctypes.c_void_p(FAKE), 1 << 40, None) == OK
    assert lib.moe_lora_linear(ctypes.byref(moelora_linear_dims(8, 8190, 28672, 32, 16)), *P,
                               ctypes.c_void_p(FAKE), 1 << 40, None) == UNSUP
    assert lib.moe_lora_linear(ctypes.byref(d), *P, ctypes.c_void_p(FAKE), 1, None) == WS
    A = [ctypes.c_void_p(FAKE)] * 6
    dd = _d()
    assert lib.moe_lora_align(ctypes.byref(dd), A[0], A[1], 0, *A[2:], ctypes.c_void_p(FAKE),
                              1 << 40, None) == INVALID                 # block_m 0
    assert lib.moe_lora_align(ctypes.byref(dd), A[0], A[1], 16, *A[2:], ctypes.c_void_p(FAKE),
                              1, None) == WS
    assert lib.moe_lora_align(ctypes.byref(dd), None, A[1], 16, *A[2:], ctypes.c_void_p(FAKE),
                              1 << 40, None) == INVALID


def test_timing_hook_host_only(lib):
    assert lib.moelora_set_timing_events(None, 0) == OK
    assert lib.moelora_set_timing_events(None, 3) == INVALID
    assert lib.moelora_set_timing_events(None, -1) == INVALID


def test_shrink_splits_plan(lib, monkeypatch):
    """The shrink items' K splits are planned on the host: their fp32 parts
    take workspace only when the items are split.  Single-CTA tiles with a
    long reduction are split by default; CTA-pair (256-token) tiles are not."""
    decode = _d()                                      # 16-token tiles, K = 2880
    prefill = _d(T=4096)                               # 256-token tiles on CTA pairs
    base = {n: binding.moelora_workspace_bytes(d) for n, d in (("decode", decode), ("prefill", prefill))}
    monkeypatch.setenv("MOELORA_SHRINK_SPLITS", "1")
    one = {n: binding.moelora_workspace_bytes(d) for n, d in (("decode", decode), ("prefill", prefill))}
    monkeypatch.setenv("MOELORA_SHRINK_SPLITS", "4")
    four = {n: binding.moelora_workspace_bytes(d) for n, d in (("decode", decode), ("prefill", prefill))}
    monkeypatch.delenv("MOELORA_SHRINK_SPLITS")
    assert base["decode"] > one["decode"]              # split by default
    assert base["prefill"] == one["prefill"]           # pairs keep one part
    assert four["decode"] > base["decode"] and four["prefill"] > one["prefill"]
    # the one- or two-phase choice needs no workspace of its own
    monkeypatch.setenv("MOELORA_TWO_PHASE", "0")
    assert binding.moelora_workspace_bytes(decode) == base["decode"]
    assert binding.moelora_workspace_bytes(_d(L=0, r=0)) < base["decode"]
