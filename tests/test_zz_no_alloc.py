"""The align entry point for callers that cannot allocate device memory.

moe_lora_align_noalloc keeps its scratch in a fixed array inside the
library instead of a caller workspace, for code that runs during CUDA-graph
capture, plug-ins without an allocator, or servers whose device memory is
all reserved by their own pool.  Its results must be identical to
moe_lora_align's (the align is integer work: bit-exact), on two calls in a
row (the shared array keeps the previous call's contents), and it must
reject sizes beyond its fixed scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.inputs import CONFIGS, make_routing

pytestmark = pytest.mark.gpu


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("name", ["decode", "prefill", "skewed"])
def test_noalloc_align_matches_workspace_align_twice(name):
    c = CONFIGS[name]
    ids, _, lo = make_routing(c, seed=0)
    ids, lo = ids.cuda(), lo.cuda()
    ref = binding.moe_lora_align(ids, lo, c.E, c.L, 16)
    first = binding.moe_lora_align_noalloc(ids, lo, c.E, c.L, 16)
    torch.cuda.synchronize()
    assert _same(ref, first)
    # a second call with other routing, then the first routing again: the
    # shared scratch keeps the previous call's contents and must not leak
    ids2, _, lo2 = make_routing(c, seed=1)
    ref2 = binding.moe_lora_align(ids2.cuda(), lo2.cuda(), c.E, c.L, 16)
    second = binding.moe_lora_align_noalloc(ids2.cuda(), lo2.cuda(), c.E, c.L, 16)
    third = binding.moe_lora_align_noalloc(ids, lo, c.E, c.L, 16)
    torch.cuda.synchronize()
    assert _same(ref2, second)
    assert _same(ref, third)


def test_noalloc_align_rejects_sizes_beyond_its_scratch():
    lib = binding.load()
    d = binding.moelora_dims(1 << 20, 1, 64, 8, 8, 16, 0)   # ~1M entries, 1088 bins
    fake = ctypes.c_void_p(0x7f0000000000)
    st = lib.moe_lora_align_noalloc(ctypes.byref(d), fake, fake, 16, fake, fake, fake, fake, None)
    assert st == -4   # MOELORA_ERR_WORKSPACE
