#!/usr/bin/env python
"""Benchmark of the fused MoE-LoRA expert layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode|prefill|skewed|tiny|dense_t1|...]

One step = one call of the whole layer (align, permute, gate_up GEMM with
its LoRA shrink/expand, down GEMM with its LoRA, combine) on one batch of
seeded synthetic input.  The default workload is the decode batch (T=16,
H=I=2880, 32 experts top-4, 8 adapters of rank 32); its weights (1.6 GB) are
larger than the 129 MB L2, so no flush is needed between steps.

Under torchrun every rank runs an independent replica on its own GPU with
its own batch (no collective on the data path); the timed region is
bracketed by a barrier and a synchronize, and the slowest rank's time
counts.  Rank 0 prints one JSON line.

With the decode batch as the headline (the default), one GPU, the other
workloads (prefill, skewed, the dense linear and the dense MLP at T = 1, 8,
64, 512, and the merged-weight fast path on the decode and skewed layers)
are timed after it, about a quarter second each, and reported under
`per_config` with their own roofline, clocks and parity.  Every timed
output is compared with the oracle over its whole batch (`parity`).

A tensor-bound kernel is rated against the burst bf16 peak when its timed
loop is shorter than 1.5 s (every default loop), else against the sustained
(power-capped) one; `roofline.peak_source` names the peak used.

--impl reference times the CPU oracle (float64 numpy) on this host's cores
on a bounded sample of the same workload; only rank 0 works under torchrun.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer routed tokens/s; % of HBM (decode) / bf16 TC (prefill) roofline"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="bounded CPU work of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the oracle comparison of the timed outputs")
    ap.add_argument("--per-config", default=None,
                    help="comma-separated workloads timed after the headline, each reported under "
                         "per_config ('none' for none; default: every other workload when the "
                         "headline is the decode batch)")
    ap.add_argument("--tuning", default=os.path.join(ROOT, "lora_mixture_experts_gb300", "tuning"),
                    help="tuned launch-choice table (file or folder); 'none' = built-in choices")
    return ap.parse_args()


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.samples = []
        self.window = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", index, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [v.strip() for v in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.01)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        note = "inside timed region"
        if not inside and self.samples:
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:2]
            inside = [s for _, s in near]
            note = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        mx = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# --------------------------------------------------------------- helpers
def reduce_max(v: float, world: int, device) -> float:
    """The slowest rank's figure (every rank gets it); a no-op on one rank."""
    if world <= 1:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each replica draws its own batch (weights and routing) from its rank."""
    return rank


def workload_name(c):
    from lora_mixture_experts_gb300.inputs import LinearCase
    if isinstance(c, LinearCase):
        return (f"{c.name}: dense multi-LoRA linear x[{c.T},{c.K}] @ W[{c.N},{c.K}]^T + LoRA "
                f"r={c.r} over {c.L} adapters")
    return (f"{c.name}: T={c.T}, H={c.H}, I={c.I}, E={c.E}, top-{c.k}, {c.L} adapters r={c.r}, "
            f"routing={c.routing}, adapters={c.adapters}")


def source_hash():
    """Hash of the GEMM and merge kernels' sources without their comments and
    blank space: a DRAM-traffic figure captured by ncu is reported only while
    the code it measured is unchanged (a comment edit keeps it)."""
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "lora_mixture_experts_gb300", "csrc")
    for n in ("gemm_tc.cu", "gemm_tc.cuh", "common.cuh", "merge.cu", "merge.cuh"):
        with open(os.path.join(d, n)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(config_name, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries
    (lines `traffic: config=... kernel=... bytes_per_launch=... source_hash=...`
    in profiles/*.md), or None if none matches the current kernel source."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    want = source_hash()
    for n in sorted(os.listdir(d)):
        if not n.endswith(".md"):
            continue
        with open(os.path.join(d, n)) as f:
            for line in f:
                if not line.startswith("traffic:"):
                    continue
                kv = dict(tok.split("=", 1) for tok in line.split()[1:] if "=" in tok)
                if (kv.get("config") == config_name and kv.get("kernel") == kernel
                        and kv.get("source_hash") == want):
                    return int(kv["bytes_per_launch"])
    return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_baseline(case, host, seconds, tokens=None):
    """Times the oracle on this host on a bounded sample; returns (tokens/s, sample text)."""
    from oracle import moe_lora_ref as ref
    from lora_mixture_experts_gb300.inputs import LinearCase
    T = case.T
    if tokens is None:
        tokens = list(range(T))
    n_done = 0
    reps = 0
    t0 = time.perf_counter()
    while True:
        if isinstance(case, LinearCase):
            y = ref.moe_lora_linear_ref(host["x"][tokens], host["lora_ids"][tokens], host["W"],
                                        host["A"], host["B"])
        else:
            y = ref.moe_lora_forward_ref(host["x"], host["topk_ids"], host["topk_weights"],
                                         host["lora_ids"], host["W_gate_up"], host["W_down"],
                                         host.get("A_gu"), host.get("B_gu"), host.get("A_d"),
                                         host.get("B_d"), tokens=tokens)
        n_done += len(tokens)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    sample = (f"{len(tokens)} of {T} tokens of the {case.name} batch per oracle call, "
              f"{reps} calls in {el:.1f} s")
    return n_done / el, sample, y


def parity_summary(gpu_rows, ref_rows):
    """The layer's acceptance figures for the timed output against the
    oracle's rows of the same tokens: relative Frobenius error (tolerance
    1e-2) and max-abs error over the oracle's RMS (tolerance 3e-2)."""
    import numpy as np
    g = gpu_rows.float().cpu().numpy().astype(np.float64)
    d = g - ref_rows
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref_rows), 1e-30))
    rms = float(np.sqrt(np.mean(ref_rows ** 2)))
    mx = float(np.abs(d).max() / max(rms, 1e-30))
    return {"tokens": int(ref_rows.shape[0]), "rel_fro": rel, "max_abs_over_rms": mx,
            "tolerance": {"rel_fro": 1e-2, "max_abs_over_rms": 3e-2},
            "pass": bool(np.all(np.isfinite(g)) and rel <= 1e-2 and mx <= 3e-2)}


def host_inputs(d):
    from lora_mixture_experts_gb300.inputs import bf16_bits
    import torch
    out = {}
    for k, v in d.items():
        out[k] = bf16_bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()
    return out


def sample_tokens(case, budget_tokens):
    import numpy as np
    if case.T <= budget_tokens:
        return list(range(case.T))
    rng = np.random.default_rng(0)
    return sorted(rng.choice(case.T, size=budget_tokens, replace=False).tolist())


def oracle_budget_tokens(case):
    # tokens per oracle call: the whole batch when it is small, else a sample
    # that keeps one call around a second
    from lora_mixture_experts_gb300.inputs import LinearCase
    if isinstance(case, LinearCase):
        return min(case.T, 64)
    return min(case.T, 64 if case.H * case.I <= 2880 * 2880 else 16)


# --------------------------------------------------------------- arms
def run_reference(args, rank, world):
    from lora_mixture_experts_gb300.inputs import CONFIGS, LinearCase, make_linear_case, make_moe_case
    if rank != 0:
        return None
    case = CONFIGS[args.config]
    d = make_linear_case(case, 0, "cpu") if isinstance(case, LinearCase) else make_moe_case(case, 0, "cpu")
    host = host_inputs(d)
    tokens = sample_tokens(case, oracle_budget_tokens(case))
    from oracle import moe_lora_ref as ref
    for _ in range(max(args.warmup, 0)):
        oracle_baseline(case, host, 0.0, tokens)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_baseline(case, host, 0.0, tokens)
        times.append(time.perf_counter() - t0)
    el = sum(times)
    value = len(tokens) * args.steps / el
    sample = f"{len(tokens)} of {case.T} tokens of the {case.name} batch per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(case), "parallelism": "host CPU (oracle)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


class _LazyBits:
    """Indexable host view of a device bf16 tensor: an index copies only that
    slice to the host (as bf16 bit patterns), so the oracle reads one
    expert's weights at a time instead of a copy of the whole set."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        from lora_mixture_experts_gb300.inputs import bf16_bits
        return bf16_bits(self.t[idx])


def oracle_full(case, d):
    """The oracle's output for every token of the batch in `d` (device
    tensors), weights read one expert at a time."""
    import torch
    from oracle import moe_lora_ref as ref
    from lora_mixture_experts_gb300.inputs import LinearCase, bf16_bits
    if isinstance(case, LinearCase):
        return ref.moe_lora_linear_ref(bf16_bits(d["x"]), d["lora_ids"].cpu().numpy(), bf16_bits(d["W"]),
                                       bf16_bits(d["A"]), bf16_bits(d["B"]))
    h = {}
    for k, v in d.items():
        if v.dtype == torch.bfloat16:
            h[k] = bf16_bits(v) if k == "x" else _LazyBits(v)
        else:
            h[k] = v.cpu().numpy()
    return ref.moe_lora_forward_ref(h["x"], h["topk_ids"], h["topk_weights"], h["lora_ids"],
                                    h["W_gate_up"], h["W_down"], h.get("A_gu"), h.get("B_gu"),
                                    h.get("A_d"), h.get("B_d"))


# a kernel timed inside a loop shorter than this is rated against the burst
# bf16 peak, a longer one against the sustained (power-capped) peak
SUSTAINED_AFTER_S = 1.5


def measure(case, args, steps, warmup, rank, world, device, peaks, sampler, e2e=True, target_s=0.25):
    """Times one workload: `steps` calls of the whole layer after `warmup`
    calls (steps=None: as many as take about target_s; device time between
    CUDA events, max over ranks), then the same
    steps with an event around every kernel of the call (the dominant
    kernel's time), then the end-to-end loop through the public API.
    Returns (result dict, output tensor, device inputs)."""
    import torch
    from lora_mixture_experts_gb300 import binding, roofline
    from lora_mixture_experts_gb300.inputs import LinearCase, make_linear_case, make_moe_case

    linear = isinstance(case, LinearCase)
    seed = rank_seed(rank)
    d = make_linear_case(case, seed=seed, device=device) if linear else make_moe_case(case, seed=seed, device=device)
    if linear:
        dims = binding.moelora_linear_dims(case.T, case.K, case.N, case.L, case.r)
        ws = binding.alloc_workspace(binding.moelora_linear_workspace_bytes(dims), device)
        out = torch.empty((case.T, case.N), dtype=torch.bfloat16, device=device)

        def fwd(x=d["x"], lo=d["lora_ids"], o=None):
            binding.moe_lora_linear(x, lo, d["W"], d["A"], d["B"], out=out if o is None else o, ws=ws)
        layer = roofline.linear_work(d["lora_ids"].cpu().numpy(), case.K, case.N, case.r)
        kernel_work = {"gemm_linear": layer}
        step_inputs = ["x", "lora_ids"]
    else:
        dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
        ws = binding.alloc_workspace(binding.moelora_workspace_bytes(dims), device)
        out = torch.empty_like(d["x"])

        def fwd(x=d["x"], ids=d["topk_ids"], w=d["topk_weights"], lo=d["lora_ids"], o=None):
            binding.moe_lora_forward(x, ids, w, lo, d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"],
                                     d["A_d"], d["B_d"], out=out if o is None else o, ws=ws)
        layer, gu, dn = roofline.moe_layer_work(d["topk_ids"].cpu().numpy(), d["lora_ids"].cpu().numpy(),
                                                case.H, case.I, case.r)
        # single-CTA tiles run both projections in one launch
        kernel_work = {"gemm_gate_up": gu, "gemm_down": dn,
                       "gemm_gate_up_down": roofline.Work(gu.bytes + dn.bytes, gu.flops + dn.flops)}
        step_inputs = ["x", "topk_ids", "topk_weights", "lora_ids"]

    fwd()
    torch.cuda.synchronize()
    status = binding.moelora_get_error(ws)
    if status != 0:
        raise RuntimeError(f"{case.name}: device status {binding.moelora_status_string(status)}")
    names = binding.moelora_last_launches()
    nl = len(names)
    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    if steps is None:
        # about `target_s` of timed calls, 20 to 2000 of them
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(3):
            fwd()
        c1.record()
        torch.cuda.synchronize()
        steps = int(min(2000, max(20, target_s * 1e3 / (c0.elapsed_time(c1) / 3))))

    K = steps
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record()
    for _ in range(K):
        fwd()
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1) / K
    ms = reduce_max(ms, world, device)

    # per-kernel device time: a second pass of K steps with an event recorded
    # on the launch stream before and after every kernel of the call (events
    # between the launches stop consecutive kernels from overlapping their
    # launch, so this pass is kept apart from the one that gives `value`)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(K)]
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record()
    for i in range(K):
        binding.moelora_set_timing_events(ev[i])
        fwd()
    p1.record()
    torch.cuda.synchronize()
    t_wall2 = time.time()
    binding.moelora_set_timing_events(None)
    ms_profiled = p0.elapsed_time(p1) / K
    clocks = sampler.summary(t_wall0, t_wall2)

    per = {}
    for i in range(K):
        for j in range(nl):
            per.setdefault(names[j], []).append(ev[i][j].elapsed_time(ev[i][j + 1]))
    # median over the steps: a step that the host delayed (events recorded
    # late) does not move the kernel's figure
    kernel_ms = {n: statistics.median(v) for n, v in per.items()}
    dom = max(kernel_work, key=lambda n: kernel_ms.get(n, 0.0))
    w = kernel_work[dom]
    region_s = K * ms / 1e3
    sustained = region_s >= SUSTAINED_AFTER_S
    bound = roofline.bound_of(w, peaks, sustained)
    dur_s = kernel_ms[dom] / 1e3
    tc_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if bound == "hbm":
        achieved, peak, unit = w.bytes / dur_s / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_name = "HBM copy"
    else:
        achieved, peak, unit = w.flops / dur_s / 1e12, peaks[tc_key], "TFLOP/s"
        peak_name = ("bf16 sustained" if sustained else "bf16 burst") + \
            f" (timed region {region_s:.2f} s)"
    traffic = load_traffic(case.name, dom)
    res = {
        "ms_per_step": ms, "steps": K, "warmup": warmup,
        "value": case.T * world / (ms / 1e3), "unit": "tokens/s",
        "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peaks['source']} ({peak_name})",
                     "algorithmic_bytes": w.bytes, "algorithmic_flops": w.flops,
                     "kernel_ms": kernel_ms[dom]},
        "layer_roofline": {"bound": roofline.bound_of(layer, peaks, sustained),
                           "t_roof_ms": 1e3 * roofline.roofline_time_s(layer, peaks, sustained),
                           "frac": 1e3 * roofline.roofline_time_s(layer, peaks, sustained) / ms,
                           "bytes": layer.bytes, "flops": layer.flops},
        "kernel_ms": kernel_ms,
        "ms_per_step_with_kernel_events": ms_profiled,
        "gpu_launches": nl * K,
        "clocks": clocks,
    }
    if e2e:
        # end to end through the public API, as a serving loop runs it: every
        # step copies its inputs from pinned host memory (packed in one
        # buffer, each at a 256-byte offset, one transfer) and reads its
        # result back.  The copies run on their own streams, into and out of
        # double buffers, so that step n+1's inputs arrive and step n-1's
        # result leaves while step n computes; events order every buffer's
        # reuse after the work that last read it.
        offs, nbytes = {}, 0
        for k in step_inputs:
            offs[k] = nbytes
            nbytes += (d[k].numel() * d[k].element_size() + 255) // 256 * 256

        def view(buf, k):
            n = d[k].numel() * d[k].element_size()
            return buf[offs[k]:offs[k] + n].view(d[k].dtype).view(d[k].shape)
        host_buf = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        dev_buf = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]
        for b in range(2):
            for k in step_inputs:
                view(host_buf[b], k).copy_(d[k].cpu())
        dev_in = [{k: view(dev_buf[b], k) for k in step_inputs} for b in range(2)]
        out_d = [out, torch.empty_like(out)]
        out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        compute = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "fwd", "out")}
        used = [False, False]

        def e2e_step(n):
            b = n & 1
            if used[b]:
                h2d.wait_event(ev["fwd"][b])          # step n-2 read dev_buf[b]
            with torch.cuda.stream(h2d):
                dev_buf[b].copy_(host_buf[b], non_blocking=True)
            ev["in"][b].record(h2d)
            compute.wait_event(ev["in"][b])
            if used[b]:
                compute.wait_event(ev["out"][b])      # step n-2's result left out_d[b]
            fwd(*[dev_in[b][k] for k in step_inputs], o=out_d[b])
            ev["fwd"][b].record(compute)
            d2h.wait_event(ev["fwd"][b])
            with torch.cuda.stream(d2h):
                out_h[b].copy_(out_d[b], non_blocking=True)
            ev["out"][b].record(d2h)
            used[b] = True
        for n in range(min(warmup, 5)):
            e2e_step(n)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for n in range(K):
            e2e_step(n)
        torch.cuda.synchronize()
        e2e_s = reduce_max((time.perf_counter() - t0) / K, world, device)
        res["e2e"] = {"value": case.T * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
                      "d2h_bytes_per_step": out.numel() * out.element_size(),
                      "pipeline": "copies on two streams, double-buffered, overlapping the next and "
                                  "previous steps' compute"}
        # the read-back is this step's result: compare it with the device output
        if not torch.equal(out_h[(K - 1) & 1], out_d[(K - 1) & 1].cpu()):
            raise RuntimeError(f"{case.name}: the end-to-end read-back differs from the device output")
    # the last timed call's output is the forward of these inputs again
    fwd()
    torch.cuda.synchronize()
    return res, out, d


def merge_parity(d, Wgu, Wd, a, experts):
    """The merged weights of `experts` against float64 W + B A of adapter a
    (one bf16 rounding allowed: |got - exact| <= 2^-8 |exact| + 1e-6)."""
    import numpy as np
    from oracle import moe_lora_ref as ref
    from lora_mixture_experts_gb300.inputs import bf16_bits
    worst = 0.0
    for e in experts:
        for W, B, A, got in ((d["W_gate_up"], d["B_gu"], d["A_gu"], Wgu), (d["W_down"], d["B_d"], d["A_d"], Wd)):
            exact = ref.as_f64(bf16_bits(W[e])) + ref.as_f64(bf16_bits(B[a, e])) @ ref.as_f64(bf16_bits(A[a, e]))
            g = ref.as_f64(bf16_bits(got[e]))
            worst = max(worst, float(np.max(np.abs(g - exact) / (2.0 ** -8 * np.abs(exact) + 1e-6))))
    return {"experts": len(experts), "worst_error_over_bound": worst, "pass": bool(worst <= 1.0)}


def measure_merge(case, peaks, sampler, target_s=0.25):
    """The merged-weight fast path (moe_lora_merge_adapter) on a workload's
    layer: one call merges one adapter into both projections of every
    expert.  HBM-bound: the bytes of merge_work per call."""
    import torch
    from lora_mixture_experts_gb300 import binding, roofline
    from lora_mixture_experts_gb300.inputs import make_moe_case
    d = make_moe_case(case, seed=0, device="cuda")
    a = case.L - 1
    Wgu = torch.empty_like(d["W_gate_up"])
    Wd = torch.empty_like(d["W_down"])

    def call():
        binding.moe_lora_merge_adapter(a, d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"], d["A_d"],
                                       d["B_d"], W_gate_up_out=Wgu, W_down_out=Wd)
    call()
    torch.cuda.synchronize()
    names = binding.moelora_last_launches()
    for _ in range(3):
        call()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    call()
    e1.record()
    torch.cuda.synchronize()
    K = int(min(2000, max(20, target_s * 1e3 / e0.elapsed_time(e1))))
    t0 = time.time()
    e0.record()
    for _ in range(K):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K)]
    for i in range(K):
        binding.moelora_set_timing_events(ev[i])
        call()
    torch.cuda.synchronize()
    binding.moelora_set_timing_events(None)
    clocks = sampler.summary(t0, time.time())
    kernel_ms = {n: statistics.median([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)])
                 for j, n in enumerate(names)}
    E, H, I, r = case.E, case.H, case.I, case.r
    gu_bytes = 2 * E * 2 * I * H * 2 + E * (r * H + 2 * I * r) * 2
    achieved = gu_bytes / (kernel_ms["merge_gate_up"] / 1e3) / 1e9
    w = roofline.merge_work(E, H, I, r)
    experts = list(range(E)) if E * (3 * I * H) <= 1 << 30 else list(range(0, E, max(1, E // 4)))[:4]
    res = {
        "workload": f"merge of one adapter into {case.name}'s layer: E={E}, H={H}, I={I}, r={r}",
        "ms_per_step": ms, "steps": K, "unit": "ms per merge",
        "roofline": {"kernel": "merge_gate_up", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": f"{peaks['source']} (HBM copy)", "algorithmic_bytes": gu_bytes,
                     "kernel_ms": kernel_ms["merge_gate_up"], "traffic": load_traffic(f"merge_{case.name}", "merge_gate_up")},
        "layer_roofline": {"bound": "hbm", "t_roof_ms": 1e3 * w.bytes / (peaks["hbm_gbs"] * 1e9),
                           "frac": 1e3 * w.bytes / (peaks["hbm_gbs"] * 1e9) / ms, "bytes": w.bytes, "flops": w.flops},
        "kernel_ms": kernel_ms, "gpu_launches": len(names) * K, "clocks": clocks,
        "parity": merge_parity(d, Wgu, Wd, a, experts),
    }
    del d, Wgu, Wd
    return res


# the workloads timed after the headline in a default run (each one's own
# line under `per_config`); the headline stays the decode batch
PER_CONFIG = ("prefill", "skewed", "dense_t1", "dense_t8", "dense_t64", "dense_t512",
              "dense_mlp_t1", "dense_mlp_t8", "dense_mlp_t64", "dense_mlp_t512",
              "merge_decode", "merge_skewed")


def run_ours(args, rank, world, device):
    import torch
    from lora_mixture_experts_gb300 import binding, roofline
    from lora_mixture_experts_gb300.inputs import CONFIGS

    binding.load(build_if_missing=True)
    tuning = None
    if args.tuning and args.tuning != "none" and os.path.exists(args.tuning):
        binding.moelora_load_tuning(args.tuning)
        tuning = os.path.relpath(args.tuning, ROOT)
    case = CONFIGS[args.config]
    peaks = roofline.load_peaks(ROOT)
    dev_index = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[device.index] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(device.index)
    sampler = ClockSampler(dev_index)
    sampler.wait_first()
    try:
        m, out, d = measure(case, args, args.steps, args.warmup, rank, world, device, peaks, sampler)
        res = {
            "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_name(case), "tokens_per_step_per_gpu": case.T,
                       "l2": "weights larger than the 129 MB L2, no flush between steps",
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "tuning": tuning or "built-in choices"},
        }
        for k in ("roofline", "layer_roofline", "kernel_ms", "ms_per_step_with_kernel_events", "e2e",
                  "gpu_launches", "clocks"):
            res[k] = m[k]
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            hostw = host_inputs({k: v for k, v in d.items()})
            tokens = sample_tokens(case, oracle_budget_tokens(case))
            v, sample, _ = oracle_baseline(case, hostw, args.cpu_seconds, tokens)
            res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                   "sample": sample}
        if rank == 0 and not args.no_parity:
            # the timed output against the oracle over the whole batch
            res["parity"] = parity_summary(out, oracle_full(case, d))
        del d, out
        per_names = [n for n in (args.per_config.split(",") if args.per_config else []) if n and n != "none"]
        if world == 1 and per_names:
            res["per_config"] = {}
            for name in per_names:
                torch.cuda.empty_cache()
                if name.startswith("merge_"):
                    res["per_config"][name] = measure_merge(CONFIGS[name[len("merge_"):]], peaks, sampler)
                    continue
                c = CONFIGS[name]
                # about a quarter second of timed calls
                m, out, d = measure(c, args, None, max(args.warmup // 10, 5), rank, world, device, peaks,
                                    sampler)
                m["workload"] = workload_name(c)
                if not args.no_parity:
                    m["parity"] = parity_summary(out, oracle_full(c, d))
                res["per_config"][name] = m
                del d, out
    finally:
        sampler.stop()
    return res


def main():
    args = parse_args()
    if args.per_config is None:
        args.per_config = ",".join(PER_CONFIG) if args.config == "decode" else "none"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.config.startswith("merge_"):
        # the merged-weight fast path on its own (one GPU; for profiling)
        from lora_mixture_experts_gb300 import binding, roofline
        from lora_mixture_experts_gb300.inputs import CONFIGS
        binding.load(build_if_missing=True)
        sampler = ClockSampler(str(device.index))
        sampler.wait_first()
        try:
            res = measure_merge(CONFIGS[args.config[len("merge_"):]], roofline.load_peaks(ROOT), sampler)
        finally:
            sampler.stop()
        print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        res = run_ours(args, rank, world, device)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
