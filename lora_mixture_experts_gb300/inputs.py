"""Seeded synthetic inputs for the fused MoE-LoRA expert layer.

This module only draws random numbers with the shapes and distributions of
the layer's workloads.  It holds none of the layer's arithmetic: the router
that produces ``topk_ids``/``topk_weights`` sits upstream of the layer, and
its top-k selection is done here only to make realistic routing inputs.
Both the CUDA path and the CPU oracle take their inputs from here.

Workloads (shapes from the multi-LoRA MoE serving blog, "Implementing
multi-LoRA for MoE in vLLM": hidden 4096 -> intermediate 11008, rank 16-64;
decode/prefill shapes of a GPT-OSS-20B-like layer, 1600-in/600-out requests
with rank 32 and 8 adapters):

* ``tiny``     T=64,  H=256,  I=512,   E=8,  top-2, 4 adapters,  r=16
* ``decode``   T=16,  H=2880, I=2880,  E=32, top-4, 8 adapters,  r=32
* ``prefill``  T=4096 (8 requests x 512 tokens, one adapter each), decode shapes
* ``skewed``   T=256, H=4096, I=11008, E=64, top-6, 16 adapters, r=64,
               Zipf(1.1) expert load, Zipf adapters with 10% of tokens at -1
* ``dense``    E=1, top-1, weight 1: x[T,8192] @ W + LoRA r=16 over 32
               adapters, N=28672, T in {1, 8, 64, 512}
* ``dense_mlp`` the whole layer at E=1, top-1, weight 1 with the dense
               shapes: H=8192, I=14336 (gate_up 8192 -> 28672, down
               14336 -> 8192), LoRA r=16 over 32 adapters, T in {1, 8, 64, 512}

Distributions: x ~ N(0,1); a weight with fan-in f ~ N(0, 1/f) (variance
1/f); A ~ N(0, 1/h_in); B ~ N(0, 1/r), nonzero.  Router logits ~ N(0,1),
softmax, top-k, renormalised.  Everything is stored as bf16 except the
routing (int32 ids, fp32 weights).

Layouts (row-major, the reduction axis contiguous):
  x[T,H]; W_gate_up[E][2I][H] (rows 0..I-1 gate, I..2I-1 up); W_down[E][H][I];
  A_gu[L][E][r][H]; B_gu[L][E][2I][r]; A_d[L][E][r][I]; B_d[L][E][H][r].
  Dense linear: x[T,K]; W[N][K]; A[L][r][K]; B[L][N][r].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

__all__ = [
    "MoECase", "LinearCase", "CONFIGS", "DENSE_T_SWEEP",
    "make_moe_case", "make_linear_case", "make_routing", "bf16_bits",
]


@dataclasses.dataclass(frozen=True)
class MoECase:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    L: int
    r: int
    routing: str = "uniform"     # "uniform" | "zipf"
    adapters: str = "uniform"    # see make_routing
    zipf_s: float = 1.1
    none_frac: float = 0.0       # fraction of tokens whose adapter is -1 (zipf)
    request_len: int = 0         # > 0: one adapter per request of this many tokens


@dataclasses.dataclass(frozen=True)
class LinearCase:
    name: str
    T: int
    K: int
    N: int
    L: int
    r: int


CONFIGS: Dict[str, object] = {
    "tiny": MoECase("tiny", T=64, H=256, I=512, E=8, k=2, L=4, r=16,
                    adapters="uniform_with_none"),
    "decode": MoECase("decode", T=16, H=2880, I=2880, E=32, k=4, L=8, r=32,
                      adapters="uniform"),
    "prefill": MoECase("prefill", T=4096, H=2880, I=2880, E=32, k=4, L=8, r=32,
                       adapters="per_request", request_len=512),
    "skewed": MoECase("skewed", T=256, H=4096, I=11008, E=64, k=6, L=16, r=64,
                      routing="zipf", adapters="zipf", none_frac=0.1),
}
DENSE_T_SWEEP = (1, 8, 64, 512)
for _t in DENSE_T_SWEEP:
    CONFIGS[f"dense_t{_t}"] = LinearCase(f"dense_t{_t}", T=_t, K=8192, N=28672, L=32, r=16)
for _t in DENSE_T_SWEEP:
    CONFIGS[f"dense_mlp_t{_t}"] = MoECase(f"dense_mlp_t{_t}", T=_t, H=8192, I=14336, E=1, k=1,
                                          L=32, r=16, adapters="uniform")
# the skewed layer with a quarter of its experts (4.3 GB of weights instead of
# 17 GB): a case small enough for multi-pass profiler captures of the same
# kernel (run with the skewed batch's 256-token tiles)
CONFIGS["skewed_e16"] = MoECase("skewed_e16", T=256, H=4096, I=11008, E=16, k=6, L=16, r=64,
                                routing="zipf", adapters="zipf", none_frac=0.1)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (exact)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def _normal_bf16(shape, std, gen, device):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # draw per leading slice to bound the fp32 temporary
    flat = out.view(-1, *shape[-2:]) if len(shape) > 2 else out.view(1, *shape)
    for i in range(flat.shape[0]):
        tmp = torch.randn(flat.shape[1:], generator=gen, device=device, dtype=torch.float32)
        flat[i].copy_(tmp.mul_(std))
    return out


def make_routing(case: MoECase, seed: int = 0):
    """Routing inputs on the CPU: (topk_ids[T,k] i32, topk_weights[T,k] f32, lora_ids[T] i32)."""
    g = torch.Generator(device="cpu").manual_seed(seed * 1000003 + 17)
    T, E, k, L = case.T, case.E, case.k, case.L
    if case.routing == "uniform":
        logits = torch.randn(T, E, generator=g, dtype=torch.float64)
        p = torch.softmax(logits, dim=-1)
        w, ids = torch.topk(p, k, dim=-1)
        w = w / w.sum(dim=-1, keepdim=True)
    elif case.routing == "zipf":
        # Gumbel-top-k over log p_e, p_e ~ (e+1)^-s: sampling k experts
        # without replacement with Zipf(s) probabilities.
        pe = torch.arange(1, E + 1, dtype=torch.float64).pow(-case.zipf_s)
        pe = pe / pe.sum()
        u = torch.rand(T, E, generator=g, dtype=torch.float64).clamp_min(1e-300)
        logits = pe.log().unsqueeze(0) - torch.log(-torch.log(u))
        top, ids = torch.topk(logits, k, dim=-1)
        w = torch.softmax(top, dim=-1)
    else:
        raise ValueError(case.routing)

    if case.adapters == "uniform":
        lora = torch.randint(0, L, (T,), generator=g)
    elif case.adapters == "uniform_with_none":
        lora = torch.randint(-1, L, (T,), generator=g)
    elif case.adapters == "per_request":
        lora = (torch.arange(T) // case.request_len) % L
    elif case.adapters == "zipf":
        pa = torch.arange(1, L + 1, dtype=torch.float64).pow(-case.zipf_s)
        lora = torch.multinomial(pa / pa.sum(), T, replacement=True, generator=g)
        none = torch.rand(T, generator=g, dtype=torch.float64) < case.none_frac
        lora = torch.where(none, torch.full_like(lora, -1), lora)
    else:
        raise ValueError(case.adapters)
    return (ids.to(torch.int32).contiguous(), w.to(torch.float32).contiguous(),
            lora.to(torch.int32).contiguous())


def make_moe_case(case: MoECase, seed: int = 0, device="cpu",
                  lora: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one MoE-LoRA layer call.  Weights are drawn on ``device``
    (a CUDA generator for the large workloads), routing always on the CPU and
    then moved, so the routing of a seed is the same on every device."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    T, H, I, E, L, r = case.T, case.H, case.I, case.E, case.L, case.r
    topk_ids, topk_w, lora_ids = make_routing(case, seed)
    d = {
        "x": _normal_bf16((T, H), 1.0, g, dev),
        "topk_ids": topk_ids.to(dev),
        "topk_weights": topk_w.to(dev),
        "lora_ids": lora_ids.to(dev),
        "W_gate_up": _normal_bf16((E, 2 * I, H), H ** -0.5, g, dev),
        "W_down": _normal_bf16((E, H, I), I ** -0.5, g, dev),
    }
    if lora:
        d["A_gu"] = _normal_bf16((L, E, r, H), H ** -0.5, g, dev)
        d["B_gu"] = _normal_bf16((L, E, 2 * I, r), r ** -0.5, g, dev)
        d["A_d"] = _normal_bf16((L, E, r, I), I ** -0.5, g, dev)
        d["B_d"] = _normal_bf16((L, E, H, r), r ** -0.5, g, dev)
    return d


def make_linear_case(case: LinearCase, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """Inputs of the dense multi-LoRA linear (one expert, top-1, weight 1)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    gc = torch.Generator(device="cpu").manual_seed(seed * 1000003 + 29)
    T, K, N, L, r = case.T, case.K, case.N, case.L, case.r
    return {
        "x": _normal_bf16((T, K), 1.0, g, dev),
        "lora_ids": torch.randint(0, L, (T,), generator=gc).to(torch.int32).to(dev),
        "W": _normal_bf16((N, K), K ** -0.5, g, dev),
        "A": _normal_bf16((L, r, K), K ** -0.5, g, dev),
        "B": _normal_bf16((L, N, r), r ** -0.5, g, dev),
    }


def small_moe_case(T, H, I, E, k, L, r, seed=0, adapters="uniform_with_none",
                   routing="uniform") -> MoECase:
    """An ad-hoc case for property tests (odd sizes, tails, degenerate shapes)."""
    return MoECase(f"adhoc_T{T}_H{H}_I{I}_E{E}_k{k}_L{L}_r{r}", T=T, H=H, I=I, E=E,
                   k=k, L=L, r=r, routing=routing, adapters=adapters,
                   none_frac=0.1 if adapters == "zipf" else 0.0)
