"""The align entry point for callers that cannot allocate device memory.

moe_lora_align_noalloc keeps its scratch in a fixed array inside the
library instead of a caller workspace, for code that runs during CUDA-graph
capture, plug-ins without an allocator, or servers whose device memory is
all reserved by their own pool.  Its results must equal the oracle's align
definition bit for bit (the align is integer work), and moe_lora_align's, on
two calls in a row (the shared array keeps the previous call's contents);
it must handle an empty batch, leave out entries with out-of-range ids as
moe_lora_align does, and reject sizes beyond its fixed scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.inputs import CONFIGS, make_routing
from oracle import moe_lora_ref as ref

pytestmark = pytest.mark.gpu


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def _matches_oracle(res, ids, lo, E, L, bm):
    s, b, seg, npp = res
    exp = ref.align_ref(ids.cpu().numpy(), lo.cpu().numpy(), E, L, bm)
    P = exp["num_post_pad"]
    assert int(npp.item()) == P
    assert np.array_equal(s[:P].cpu().numpy(), exp["sorted_ids"])
    assert np.array_equal(b[:P // bm].cpu().numpy(), exp["blk_expert"])
    assert np.array_equal(seg.cpu().numpy(), exp["seg_off"])
    assert bool((s[P:] == ids.numel()).all())


@pytest.mark.parametrize("name", ["decode", "prefill", "skewed"])
def test_noalloc_align_matches_oracle_and_workspace_align_twice(name):
    c = CONFIGS[name]
    ids, _, lo = make_routing(c, seed=0)
    ids, lo = ids.cuda(), lo.cuda()
    with_ws = binding.moe_lora_align(ids, lo, c.E, c.L, 16)
    first = binding.moe_lora_align_noalloc(ids, lo, c.E, c.L, 16)
    torch.cuda.synchronize()
    _matches_oracle(first, ids, lo, c.E, c.L, 16)
    assert _same(with_ws, first)
    # a second call with other routing, then the first routing again: the
    # shared scratch keeps the previous call's contents and must not leak
    ids2, _, lo2 = make_routing(c, seed=1)
    ids2, lo2 = ids2.cuda(), lo2.cuda()
    second = binding.moe_lora_align_noalloc(ids2, lo2, c.E, c.L, 16)
    third = binding.moe_lora_align_noalloc(ids, lo, c.E, c.L, 16)
    torch.cuda.synchronize()
    _matches_oracle(second, ids2, lo2, c.E, c.L, 16)
    _matches_oracle(third, ids, lo, c.E, c.L, 16)


def test_noalloc_align_empty_batch():
    # T = 0: no entries, no blocks, every segment offset 0
    ids = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    lo = torch.empty((0,), dtype=torch.int32, device="cuda")
    res = binding.moe_lora_align_noalloc(ids, lo, 8, 3, 16)
    torch.cuda.synchronize()
    assert int(res[3].item()) == 0
    assert bool((res[2] == 0).all())
    # and a normal call right after it
    c = CONFIGS["tiny"]
    ids, _, lo = make_routing(c, seed=0)
    res = binding.moe_lora_align_noalloc(ids.cuda(), lo.cuda(), c.E, c.L, 16)
    torch.cuda.synchronize()
    _matches_oracle(res, ids, lo, c.E, c.L, 16)


def test_noalloc_align_leaves_out_bad_ids():
    # entries whose expert or adapter id is out of range are left out of the
    # order, as moe_lora_align leaves them out
    ids = torch.tensor([[0, 1], [1, 7], [2, 0]], dtype=torch.int32, device="cuda")
    lo = torch.tensor([0, -1, 5], dtype=torch.int32, device="cuda")   # 7 >= E, 5 >= L
    s, b, seg, npp = binding.moe_lora_align_noalloc(ids, lo, 4, 2, 4)
    with_ws = binding.moe_lora_align(ids, lo, 4, 2, 4)
    torch.cuda.synchronize()
    assert _same((s, b, seg, npp), with_ws)
    P = int(npp.item())
    kept = sorted(int(v) for v in s[:P].cpu() if int(v) != ids.numel())
    assert kept == [0, 1, 2]          # token 0's two entries and token 1's expert 1


def test_noalloc_align_rejects_sizes_beyond_its_scratch():
    lib = binding.load()
    d = binding.moelora_dims(1 << 20, 1, 64, 8, 8, 16, 0)   # ~1M entries, 1088 bins
    fake = ctypes.c_void_p(0x7f0000000000)
    st = lib.moe_lora_align_noalloc(ctypes.byref(d), fake, fake, 16, fake, fake, fake, fake, None)
    assert st == -4   # MOELORA_ERR_WORKSPACE
