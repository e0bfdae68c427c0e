"""Algorithmic bytes and FLOPs of one layer call, counted from the routing of
the actual instance (host-side measurement logic, not part of the layer).

Per-unit figures (bf16 = 2 bytes):
  * every expert touched by at least one routed pair reads its gate_up
    weight (2I x H) and down weight (H x I) once;
  * every (expert, adapter >= 0) pair touched reads A_gu (r x H), B_gu
    (2I x r), A_d (r x I), B_d (H x r) once;
  * x is read once per token and out written once; routing: 8 bytes per
    (token, j) entry + 4 bytes per token id.
  * FLOPs: 2 * (2I*H + I*H) per routed pair for the base projections and
    2 * (H*r + r*2I + I*r + r*H) per routed pair with an adapter; padding
    rows are not credited.
Per-kernel figures (used for the dominant kernel's roofline):
  * gate_up phase: its weights + LoRA (A_gu, B_gu) + x rows per routed pair
    (T*k*H*2, gathered) + act written (T*k*I*2);
  * down phase: its weights + LoRA (A_d, B_d) + act read (T*k*I*2) + per-pair
    outputs written in fp32 (T*k*H*4).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np


@dataclass
class Work:
    bytes: float
    flops: float


def _touched(topk_ids, lora_ids):
    ids = np.asarray(topk_ids).reshape(len(lora_ids), -1)
    lo = np.asarray(lora_ids)
    experts = np.unique(ids)
    la = np.repeat(lo, ids.shape[1])
    e = ids.reshape(-1)
    m = la >= 0
    pairs_ea = np.unique(e[m] * 1_000_003 + la[m]) if m.any() else np.array([])
    return len(experts), len(pairs_ea), int(m.sum())


def moe_layer_work(topk_ids, lora_ids, H, I, r):
    """(layer, gate_up phase, down phase) algorithmic work of one call."""
    T, k = np.asarray(topk_ids).shape
    n_e, n_ea, n_lp = _touched(topk_ids, lora_ids)
    npairs = T * k
    w_gu = n_e * 2 * I * H * 2 + n_ea * (r * H + 2 * I * r) * 2
    w_d = n_e * H * I * 2 + n_ea * (r * I + H * r) * 2
    f_gu = npairs * 2 * (2 * I * H) + n_lp * 2 * (H * r + r * 2 * I)
    f_d = npairs * 2 * (H * I) + n_lp * 2 * (I * r + r * H)
    layer = Work(w_gu + w_d + 2 * T * H * 2 + T * k * 8 + T * 4, f_gu + f_d)
    gu = Work(w_gu + npairs * H * 2 + npairs * I * 2, f_gu)
    dn = Work(w_d + npairs * I * 2 + npairs * H * 4, f_d)
    return layer, gu, dn


def linear_work(lora_ids, K, N, r):
    T = len(lora_ids)
    lo = np.asarray(lora_ids)
    n_a = len(np.unique(lo[lo >= 0]))
    n_lp = int((lo >= 0).sum())
    b = N * K * 2 + n_a * (r * K + N * r) * 2 + T * K * 2 + T * N * 2 + T * 4
    f = T * 2 * N * K + n_lp * 2 * (K * r + r * N)
    return Work(b, f)


def merge_work(E, H, I, r):
    """The merged-weight fast path for one adapter (W' = W + B A, both
    projections): every base weight read once and its merged copy written
    once, the adapter's A and B read once; 2r FLOP per merged element."""
    w = E * (2 * I * H + H * I)
    lora = E * (r * H + 2 * I * r + r * I + H * r)
    return Work(2 * w * 2 + lora * 2, 2 * r * w)


def load_peaks(root: str):
    """Measured peaks (copy bandwidth, cuBLAS bf16) if present, else the
    fallback figures of an earlier GB300 measurement."""
    path = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def roofline_time_s(w: Work, peaks, sustained=False):
    tc = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"] * 1e12
    return max(w.bytes / (peaks["hbm_gbs"] * 1e9), w.flops / tc)


def bound_of(w: Work, peaks, sustained=False):
    tc = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"] * 1e12
    return "hbm" if w.bytes / (peaks["hbm_gbs"] * 1e9) >= w.flops / tc else "tensor"
