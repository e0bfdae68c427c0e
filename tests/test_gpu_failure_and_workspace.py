"""Failure detection and workspace independence on the GPU, through the C ABI.

* A bounded wait that runs out: MOELORA_FAULT_INJECT=shrink_wait makes the
  first GEMM phase of a call wait for shrink completions that never come
  (a counter target no item reaches).  The wait gives up after the library's
  2 s limit, the kernel winds down (copies and MMAs in flight drained, TMEM
  freed), the call's status reads MOELORA_ERR_TIMEOUT, and the next call on
  the same workspace and stream is correct.  Covered for unpaired tiles,
  256-row tiles on CTA pairs, and the dense linear.  Nothing faults, traps
  or hangs.
* A workspace full of 0xFF bytes (NaN for the float buffers, -1 for the
  integer ones) gives bit-identical results to a zeroed one: no kernel reads
  a workspace byte that the same call did not write first.
"""
import time

import numpy as np
import pytest
import torch

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.inputs import CONFIGS, make_moe_case, small_moe_case
from oracle import moe_lora_ref as ref

from _parity import compare, np_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
TIMEOUT = -7


def _forward(d, ws):
    return binding.moe_lora_forward(d["x"], d["topk_ids"], d["topk_weights"], d["lora_ids"],
                                    d["W_gate_up"], d["W_down"], d.get("A_gu"), d.get("B_gu"),
                                    d.get("A_d"), d.get("B_d"), ws=ws)


def _oracle(d):
    n = np_inputs(d)
    return ref.moe_lora_forward_ref(n["x"], n["topk_ids"], n["topk_weights"], n["lora_ids"],
                                    n["W_gate_up"], n["W_down"], n.get("A_gu"), n.get("B_gu"),
                                    n.get("A_d"), n.get("B_d"))


def _moe_case(paired):
    # tiny: 16-row tiles on single CTAs; 300 rows per expert: 256-row tiles on CTA pairs
    c = small_moe_case(600, 256, 200, 2, 1, 3, 32) if paired else CONFIGS["tiny"]
    return make_moe_case(c, seed=4, device=DEV)


def _linear_case():
    g = torch.Generator(device=DEV).manual_seed(8)
    T, K, N, L, r = 45, 200, 264, 3, 32
    return dict(x=torch.randn(T, K, generator=g, device=DEV).bfloat16(),
                W=(torch.randn(N, K, generator=g, device=DEV) * K ** -0.5).bfloat16(),
                A=(torch.randn(L, r, K, generator=g, device=DEV) * K ** -0.5).bfloat16(),
                B=(torch.randn(L, N, r, generator=g, device=DEV) * r ** -0.5).bfloat16(),
                lora_ids=torch.randint(-1, L, (T,), generator=g, device=DEV).int())


def _linear(d, ws):
    return binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"], ws=ws)


def _linear_ws(d):
    T, K = d["x"].shape
    dims = binding.moelora_linear_dims(T, K, d["W"].shape[0], d["A"].shape[0], d["A"].shape[1])
    return binding.alloc_workspace(binding.moelora_linear_workspace_bytes(dims))


def _moe_ws(d):
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
    return binding.alloc_workspace(binding.moelora_workspace_bytes(dims))


def _run_timed_out(monkeypatch, call):
    monkeypatch.setenv("MOELORA_FAULT_INJECT", "shrink_wait")
    t0 = time.perf_counter()
    try:
        status = call()
    finally:
        monkeypatch.delenv("MOELORA_FAULT_INJECT")
    return status, time.perf_counter() - t0


@pytest.mark.parametrize("paired", [False, True], ids=["single_cta_tiles", "cta_pair_tiles"])
def test_wait_runs_out_then_next_call_is_correct(monkeypatch, paired):
    d = _moe_case(paired)
    ws = _moe_ws(d)

    def call():
        _forward(d, ws)
        return binding.moelora_get_error(ws)   # synchronises the stream
    status, seconds = _run_timed_out(monkeypatch, call)
    assert status == TIMEOUT, binding.moelora_status_string(status)
    assert seconds > 1.5, seconds              # the 2 s limit ran out, nothing returned early
    out = _forward(d, ws)
    assert binding.moelora_get_error(ws) == 0
    ok, msg = compare(out, _oracle(d), "after a timed-out call")
    assert ok, msg


def test_linear_wait_runs_out_then_next_call_is_correct(monkeypatch):
    d = _linear_case()
    ws = _linear_ws(d)

    def call():
        _linear(d, ws)
        return binding.moelora_get_error(ws)
    status, seconds = _run_timed_out(monkeypatch, call)
    assert status == TIMEOUT, binding.moelora_status_string(status)
    assert seconds > 1.5, seconds
    out = _linear(d, ws)
    assert binding.moelora_get_error(ws) == 0
    n = np_inputs({k: d[k] for k in ("x", "W", "A", "B")})
    exp = ref.moe_lora_linear_ref(n["x"], d["lora_ids"].cpu().numpy(), n["W"], n["A"], n["B"])
    ok, msg = compare(out, exp, "linear after a timed-out call")
    assert ok, msg


@pytest.mark.parametrize("paired", [False, True], ids=["single_cta_tiles", "cta_pair_tiles"])
def test_poisoned_workspace_gives_identical_results(paired):
    d = _moe_case(paired)
    ws = _moe_ws(d)
    ws.zero_()
    clean = _forward(d, ws).clone()
    assert binding.moelora_get_error(ws) == 0
    ws.fill_(0xFF)
    poisoned = _forward(d, ws).clone()
    assert binding.moelora_get_error(ws) == 0
    assert torch.equal(clean, poisoned)
    assert not torch.isnan(poisoned.float()).any()


def test_poisoned_workspace_linear():
    d = _linear_case()
    ws = _linear_ws(d)
    ws.zero_()
    clean = _linear(d, ws).clone()
    ws.fill_(0xFF)
    poisoned = _linear(d, ws).clone()
    assert binding.moelora_get_error(ws) == 0
    assert torch.equal(clean, poisoned)
