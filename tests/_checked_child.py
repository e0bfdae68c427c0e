"""Child process of tests/test_gpu_checked_build.py: runs a fixed set of
layer calls with whichever library MOELORA_LIBRARY names and saves every
output and device status to the file given as argv[1]."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from lora_mixture_experts_gb300 import binding  # noqa: E402
from lora_mixture_experts_gb300.inputs import (CONFIGS, make_linear_case,  # noqa: E402
                                               make_moe_case, small_moe_case)

DEV = "cuda:0"


def forward(d):
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d.get("A_gu"))
    ws = binding.alloc_workspace(binding.moelora_workspace_bytes(dims), DEV)
    ws.fill_(0xFF)
    out = binding.moe_lora_forward(d["x"], d["topk_ids"], d["topk_weights"], d["lora_ids"],
                                   d["W_gate_up"], d["W_down"], d.get("A_gu"), d.get("B_gu"),
                                   d.get("A_d"), d.get("B_d"), ws=ws)
    return out.clone(), binding.moelora_get_error(ws)


def linear(d):
    T, K = d["x"].shape
    dims = binding.moelora_linear_dims(T, K, d["W"].shape[0], d["A"].shape[0], d["A"].shape[1])
    ws = binding.alloc_workspace(binding.moelora_linear_workspace_bytes(dims), DEV)
    ws.fill_(0xFF)
    out = binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"], ws=ws)
    return out.clone(), binding.moelora_get_error(ws)


def main(path):
    binding.load(build_if_missing=False)
    binding.moelora_load_tuning(os.path.join(ROOT, "lora_mixture_experts_gb300", "tuning"))
    res = {"library": binding.library_path()}
    for name in ("tiny", "decode", "dense_mlp_t8"):
        res[name] = forward(make_moe_case(CONFIGS[name], seed=0, device=DEV))
    for shape in [(600, 256, 200, 2, 1, 3, 32), (300, 264, 264, 8, 2, 4, 16), (1100, 128, 64, 8, 2, 3, 16)]:
        res[str(shape)] = forward(make_moe_case(small_moe_case(*shape), seed=1, device=DEV))
    res["dense_t64"] = linear(make_linear_case(CONFIGS["dense_t64"], seed=0, device=DEV))
    # out-of-range ids: the align's own check, not a failed device check
    d = make_moe_case(CONFIGS["tiny"], seed=2, device=DEV)
    d["topk_ids"][3, 0] = 99
    res["bad_id"] = forward(d)
    torch.save(res, path)


if __name__ == "__main__":
    main(sys.argv[1])
