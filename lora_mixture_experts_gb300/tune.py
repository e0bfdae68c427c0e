"""Sweeps the launch choices of the layer on the current GPU and writes
tuning tables for ``moelora_load_tuning``.

    python -m lora_mixture_experts_gb300.tune [--out-dir DIR] [--families moe,skewed,...]

A family is one layer shape (k, E, H, I, L, r, or K, N, L, r for the dense
linear) swept over a ladder of batch sizes T.  At every T of the ladder each
candidate (token tile tn, K split, on single-CTA tiles one or two launches
for the projections, and on a one-expert layer a K split of the gate_up
phase) is forced with a one-line table and the whole layer call is timed
with CUDA events.  The ladder then becomes batch-size
buckets: the bucket of a sampled T reaches halfway (geometrically) to its
neighbours, the last one to any larger T, and neighbouring buckets with the
same winner merge into one `T=lo-hi` line.  A bucket whose winner is within
the timing noise of the built-in choice gets no line (the built-in choice
applies there).  (The multi-LoRA MoE blog tunes its kernels' block sizes and
split factors per workload size and loads the tuned configs from a folder:
"Kernel config tuning".)
"""
from __future__ import annotations

import argparse
import dataclasses
import math
import os
import tempfile

import torch

from . import binding
from .inputs import CONFIGS, LinearCase, MoECase, make_linear_case, make_moe_case

TILES = (16, 32, 64, 128, 256)
# a candidate replaces the built-in choice only if it is faster by more than this
KEEP_MARGIN = 0.005
T_MAX = 1 << 20


@dataclasses.dataclass(frozen=True)
class Family:
    name: str
    base: object           # a workload of the family (its T is replaced)
    ladder: tuple          # batch sizes swept


FAMILIES = {
    # the decode and prefill workloads' layer (GPT-OSS-20B-like shapes)
    "moe": Family("moe", CONFIGS["decode"], (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)),
    # the Zipf-routed large-expert layer
    "skewed": Family("skewed", CONFIGS["skewed"], (32, 64, 128, 256, 512, 1024)),
    "dense_linear": Family("dense_linear", CONFIGS["dense_t1"], (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024)),
    "dense_mlp": Family("dense_mlp", CONFIGS["dense_mlp_t1"], (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)),
}


def case_at(fam: Family, T: int):
    """The family's workload at batch size T (prefill-style requests of 512
    tokens, one adapter each, from T = 512 up on the decode/prefill layer)."""
    c = fam.base
    if isinstance(c, LinearCase):
        return dataclasses.replace(c, name=f"{fam.name}_t{T}", T=T)
    if fam.name == "moe" and T >= 512:
        return dataclasses.replace(CONFIGS["prefill"], name=f"{fam.name}_t{T}", T=T)
    return dataclasses.replace(c, name=f"{fam.name}_t{T}", T=T)


def buckets(ladder):
    """[lo, hi] batch-size range of each ladder point: halfway in log scale
    to the neighbours, from 1 up to T_MAX."""
    out = []
    for i, t in enumerate(ladder):
        lo = 1 if i == 0 else int(math.floor(math.sqrt(ladder[i - 1] * t))) + 1
        hi = T_MAX if i == len(ladder) - 1 else int(math.floor(math.sqrt(t * ladder[i + 1])))
        out.append((lo, hi))
    return out


def merge_lines(shape_key: str, picks):
    """picks: per ladder point (lo, hi, choice or None).  Neighbouring
    buckets with the same choice merge; None (built-in kept) gives no line."""
    lines = []
    cur = None
    for lo, hi, ch in picks:
        if cur is not None and ch == cur[2] and ch is not None:
            cur = (cur[0], hi, ch)
            continue
        if cur is not None and cur[2] is not None:
            lines.append((cur[0], cur[1], cur[2]))
        cur = (lo, hi, ch)
    if cur is not None and cur[2] is not None:
        lines.append(cur)
    return [f"{shape_key.replace('T=@', f'T={lo}-{hi}')} {ch}" for lo, hi, ch in lines]


def _time(fn, budget_ms=60.0):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    iters = int(min(100, max(10, budget_ms / max(e0.elapsed_time(e1), 1e-3))))
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def _shape_key(case) -> str:
    if isinstance(case, LinearCase):
        return f"linear T=@ K={case.K} N={case.N} L={case.L} r={case.r}"
    return f"moe T=@ k={case.k} E={case.E} H={case.H} I={case.I} L={case.L} r={case.r}"


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


def best_choice(case, device, cand_file, log=print):
    """(built-in ms, best ms, best choice text) at one batch size."""
    d = (make_linear_case(case, 0, device) if isinstance(case, LinearCase)
         else make_moe_case(case, 0, device))
    make = _runner(case, d, device)
    binding.moelora_load_tuning(None)
    default_ms = _time(make())
    best = None
    line0 = _shape_key(case).replace("T=@", f"T={case.T}")
    for tn in TILES:
        if tn > 16 and tn // 2 >= max(case.T * getattr(case, "k", 1), 16):
            continue     # a tile more than twice the whole batch only adds padding
        # both projections in one launch is an option on single-CTA tiles,
        # and on a one-expert layer a K-split gate_up phase
        phase_opts = (1, 2) if (not isinstance(case, LinearCase) and tn < 256) else (0,)
        gu_opts = (1, 2, 3) if (not isinstance(case, LinearCase) and tn < 256 and case.E == 1) else (1,)
        for ks, ph, gks in [(ks, ph, g) for ks in ((1,) if tn == 256 else (1, 2, 3, 4))
                            for ph in phase_opts for g in gu_opts]:
                choice = (f"tn={tn} ksplit={ks}" + (f" phases={ph}" if ph else "") +
                          (f" guksplit={gks}" if gks > 1 else ""))
                with open(cand_file, "w") as f:
                    f.write(f"{line0} {choice}\n")
                binding.moelora_load_tuning(cand_file)
                ms = _time(make())
                log(f"{case.name}: {choice}: {ms:.4f} ms")
                if best is None or ms < best[0]:
                    best = (ms, choice)
    binding.moelora_load_tuning(None)
    del d
    torch.cuda.empty_cache()
    return default_ms, best[0], best[1]


def sweep_family(fam: Family, device="cuda", log=print):
    picks, notes = [], []
    with tempfile.TemporaryDirectory() as tmp:
        cand_file = os.path.join(tmp, "candidate.cfg")
        for (lo, hi), T in zip(buckets(fam.ladder), fam.ladder):
            case = case_at(fam, T)
            default_ms, ms, choice = best_choice(case, device, cand_file, log)
            if ms < (1.0 - KEEP_MARGIN) * default_ms:
                picks.append((lo, hi, choice))
                notes.append(f"# T={T} (bucket {lo}-{hi}): {choice} {ms:.4f} ms "
                             f"(built-in choice {default_ms:.4f} ms)")
            else:   # within the timing noise of the built-in choice: keep it
                picks.append((lo, hi, None))
                notes.append(f"# T={T} (bucket {lo}-{hi}): built-in choice kept ({default_ms:.4f} ms; "
                             f"best candidate {choice} {ms:.4f} ms)")
    return merge_lines(_shape_key(case_at(fam, fam.ladder[0])), picks), notes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out-dir", default=os.path.join(os.path.dirname(__file__), "tuning"))
    ap.add_argument("--families", default=",".join(FAMILIES))
    args = ap.parse_args()
    os.makedirs(args.out_dir, exist_ok=True)
    binding.load()
    for name in args.families.split(","):
        fam = FAMILIES[name]
        lines, notes = sweep_family(fam)
        text = [f"# Launch choices for the {name} layer family, tuned on this GPU by "
                "lora_mixture_experts_gb300.tune",
                f"# device: {torch.cuda.get_device_name()}",
                "# batch-size buckets (first matching line wins; T outside every line: built-in choice)"]
        text += lines + notes
        with open(os.path.join(args.out_dir, f"gb300_{name}.cfg"), "w") as f:
            f.write("\n".join(text) + "\n")
        print("\n".join(text), flush=True)


if __name__ == "__main__":
    main()
