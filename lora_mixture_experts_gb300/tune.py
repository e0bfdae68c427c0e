"""Sweeps the launch choices of the layer per workload on the current GPU
and writes a tuning table for ``moelora_load_tuning``.

    python -m lora_mixture_experts_gb300.tune [--out FILE] [--configs decode,prefill,...]

For every workload and every candidate (token tile tn, K split, and on
single-CTA tiles one or two launches for the projections) it forces the
candidate with a one-line table, times the whole layer call with CUDA events
and keeps the fastest; the table lines match the workload's exact shape.
(The multi-LoRA MoE blog tunes its kernels' block sizes and split factors per
workload and loads the tuned configs from a folder: "Kernel config tuning".)
"""
from __future__ import annotations

import argparse
import os
import tempfile

import torch

from . import binding
from .inputs import CONFIGS, LinearCase, make_linear_case, make_moe_case

TILES = (16, 32, 64, 128, 256)
# a candidate replaces the built-in choice only if it is faster by more than this
KEEP_MARGIN = 0.005


def _time(fn, warmup=5, iters=100):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def _shape_line(case) -> str:
    if isinstance(case, LinearCase):
        return f"linear T={case.T} K={case.K} N={case.N} L={case.L} r={case.r}"
    return f"moe T={case.T} k={case.k} E={case.E} H={case.H} I={case.I} L={case.L} r={case.r}"


def _runner(case, d, device):
    if isinstance(case, LinearCase):
        dims = binding.moelora_linear_dims(case.T, case.K, case.N, case.L, case.r)
        out = torch.empty((case.T, case.N), dtype=torch.bfloat16, device=device)

        def make():
            ws = binding.alloc_workspace(binding.moelora_linear_workspace_bytes(dims), device)
            return lambda: binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"],
                                                   out=out, ws=ws)
        return make
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
    out = torch.empty_like(d["x"])

    def make():
        ws = binding.alloc_workspace(binding.moelora_workspace_bytes(dims), device)
        return lambda: binding.moe_lora_forward(d["x"], d["topk_ids"], d["topk_weights"],
                                                d["lora_ids"], d["W_gate_up"], d["W_down"],
                                                d["A_gu"], d["B_gu"], d["A_d"], d["B_d"],
                                                out=out, ws=ws)
    return make


def sweep(names, out_path, device="cuda", log=print):
    lines = ["# Launch choices tuned on this GPU by lora_mixture_experts_gb300.tune",
             f"# device: {torch.cuda.get_device_name(device)}"]
    with tempfile.TemporaryDirectory() as tmp:
        cand_file = os.path.join(tmp, "candidate.cfg")
        for name in names:
            case = CONFIGS[name]
            d = (make_linear_case(case, 0, device) if isinstance(case, LinearCase)
                 else make_moe_case(case, 0, device))
            make = _runner(case, d, device)
            binding.moelora_load_tuning(None)
            default_ms = _time(make())
            best = None
            for tn in TILES:
                # both projections in one launch is an option on single-CTA tiles
                phase_opts = (1, 2) if (not isinstance(case, LinearCase) and tn < 256) else (0,)
                for ks in (1, 2, 3, 4):
                    for ph in phase_opts:
                        extra = f" phases={ph}" if ph else ""
                        with open(cand_file, "w") as f:
                            f.write(f"{_shape_line(case)} tn={tn} ksplit={ks}{extra}\n")
                        binding.moelora_load_tuning(cand_file)
                        ms = _time(make())
                        log(f"{name}: tn={tn} ksplit={ks}{extra}: {ms:.4f} ms")
                        if best is None or ms < best[0]:
                            best = (ms, tn, ks, extra)
            binding.moelora_load_tuning(None)
            ms, tn, ks, extra = best
            if ms < (1.0 - KEEP_MARGIN) * default_ms:
                lines.append(f"{_shape_line(case)} tn={tn} ksplit={ks}{extra}   "
                             f"# {name}: {ms:.4f} ms (built-in choice {default_ms:.4f} ms)")
            else:   # within the timing noise of the built-in choice: keep it
                lines.append(f"# {name}: built-in choice kept ({default_ms:.4f} ms; "
                             f"best candidate tn={tn} ksplit={ks}{extra} {ms:.4f} ms)")
            del d
            torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return lines


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(os.path.dirname(__file__), "tuning", "gb300.cfg"))
    ap.add_argument("--configs", default="decode,prefill,skewed,dense_t1,dense_t8,dense_t64,dense_t512")
    args = ap.parse_args()
    os.makedirs(os.path.dirname(os.path.abspath(args.out)), exist_ok=True)
    binding.load()
    for line in sweep(args.configs.split(","), args.out):
        print(line)


if __name__ == "__main__":
    main()
