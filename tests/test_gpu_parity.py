"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

* align: bit-exact against the oracle's definition for every workload's
  routing and for edge cases (block_m 1..128, empty experts, all tokens on one
  expert, adapters absent);
* forward: every workload at full size, every token of the batch compared
  element by element with the oracle (tiny, decode, prefill, skewed, the
  dense linear and the dense MLP at T = 1, 8, 64, 512, in the built-in and
  the tuned launch configuration); random small shapes with ragged tails (H
  not a multiple of 128, I not a multiple of 64, T = 1, k = E, every LoRA
  rank, no LoRA);
* determinism, CUDA-graph capture/replay, and the device-side bad-index flag.
"""
import numpy as np
import pytest
import torch

from lora_mixture_experts_gb300 import binding
from lora_mixture_experts_gb300.inputs import (CONFIGS, DENSE_T_SWEEP, make_linear_case,
                                               make_moe_case, make_routing, small_moe_case)
from oracle import moe_lora_ref as ref

from _parity import compare, np_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu_forward(d, **kw):
    return binding.moe_lora_forward(d["x"], d["topk_ids"], d["topk_weights"], d["lora_ids"],
                                    d["W_gate_up"], d["W_down"], d.get("A_gu"), d.get("B_gu"),
                                    d.get("A_d"), d.get("B_d"), **kw)


def _oracle_forward(n, tokens=None):
    return ref.moe_lora_forward_ref(n["x"], n["topk_ids"], n["topk_weights"], n["lora_ids"],
                                    n["W_gate_up"], n["W_down"], n.get("A_gu"), n.get("B_gu"),
                                    n.get("A_d"), n.get("B_d"), tokens=tokens)


# ------------------------------------------------------------------ align
def _check_align(topk_ids, lora_ids, E, L, bm):
    s, b, seg, npp = binding.moe_lora_align(topk_ids.to(DEV), lora_ids.to(DEV), E, L, bm)
    torch.cuda.synchronize()
    exp = ref.align_ref(topk_ids.numpy(), lora_ids.numpy(), E, L, bm)
    P = exp["num_post_pad"]
    assert int(npp.item()) == P
    assert np.array_equal(s[:P].cpu().numpy(), exp["sorted_ids"])
    assert np.array_equal(b[:P // bm].cpu().numpy(), exp["blk_expert"])
    assert np.array_equal(seg.cpu().numpy(), exp["seg_off"])
    n = topk_ids.numel()
    assert bool((s[P:] == n).all())


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed"])
@pytest.mark.parametrize("bm", [1, 16, 128])
def test_align_workloads(name, bm):
    c = CONFIGS[name]
    ids, _, lora = make_routing(c, seed=0)
    _check_align(ids, lora, c.E, c.L, bm)


def test_align_edge_cases():
    g = torch.Generator().manual_seed(3)
    # all tokens on expert 2 of 5, every adapter -1
    _check_align(torch.full((37, 1), 2, dtype=torch.int32), torch.full((37,), -1, dtype=torch.int32), 5, 3, 8)
    # one token
    _check_align(torch.tensor([[4, 1]], dtype=torch.int32), torch.tensor([0], dtype=torch.int32), 6, 1, 16)
    # more entries than one align chunk, with empty experts and L = 0
    ids = torch.randint(0, 3, (700, 2), generator=g, dtype=torch.int32) * 3
    _check_align(ids, torch.full((700,), -1, dtype=torch.int32), 9, 0, 4)
    # many bins
    ids = torch.randint(0, 64, (900, 3), generator=g, dtype=torch.int32)
    lo = torch.randint(-1, 40, (900,), generator=g, dtype=torch.int32)
    _check_align(ids, lo, 64, 40, 32)


def test_align_large_shapes():
    g = torch.Generator().manual_seed(9)
    # more bins than the single-CTA path holds (256 experts x 33 adapter bins)
    ids = torch.randint(0, 256, (300, 2), generator=g, dtype=torch.int32)
    lo = torch.randint(-1, 32, (300,), generator=g, dtype=torch.int32)
    _check_align(ids, lo, 256, 32, 16)
    # 65536 entries: 256 chunks through the three-kernel path
    c = small_moe_case(8192, 64, 64, 256, 8, 4, 16, routing="zipf")
    ids, _, lo = make_routing(c, seed=2)
    _check_align(ids, lo, 256, 4, 16)


def test_align_maximum_bins():
    """E = 1024 experts and L = 10 adapters: E*(L+1) = 11264 bins, the most the
    library accepts; a tiny batch (too many bins for the single-CTA path) and
    a 16384-entry batch."""
    g = torch.Generator().manual_seed(11)
    for T, k in ((5, 3), (2048, 8)):
        ids = torch.stack([torch.randperm(1024, generator=g)[:k] for _ in range(T)]).to(torch.int32)
        lo = torch.randint(-1, 10, (T,), generator=g, dtype=torch.int32)
        _check_align(ids, lo, 1024, 10, 16)


def test_align_bad_index_flag():
    ids = torch.tensor([[0, 1], [1, 7]], dtype=torch.int32, device=DEV)
    lo = torch.tensor([0, -1], dtype=torch.int32, device=DEV)
    d = binding.moelora_dims(2, 2, 4, 8, 8, 2, 0)
    ws = binding.alloc_workspace(binding.moelora_align_workspace_bytes(d))
    s, b, seg, npp = binding.moe_lora_align(ids, lo, 4, 2, 4, ws=ws)
    assert binding.moelora_get_error(ws) == -6
    assert int(npp.item()) == 8           # three valid entries: expert 0 (1) and 1 (2), padded to 4


# ------------------------------------------------------------------ forward
# oracle outputs of the full-size workloads, shared by the tests that run one
# workload in several launch configurations
_ORACLE = {}


def _large(d):
    return sum(v.numel() * v.element_size() for v in d.values()) > (256 << 20)


def _run_parity(d, tokens=None, what="", key=None):
    """The layer on the GPU against the oracle: every token of the batch
    (or the given tokens), element by element.  Large weights are copied to
    the host one expert at a time as the oracle reaches them."""
    out = _gpu_forward(d)
    torch.cuda.synchronize()
    if key is not None and key in _ORACLE:
        exp = _ORACLE[key]
    else:
        n = np_inputs(d, lazy=tokens is not None or _large(d))
        exp = _oracle_forward(n, tokens)
        if key is not None:
            _ORACLE[key] = exp
    got = out if tokens is None else out[torch.as_tensor(tokens, device=out.device)]
    ok, msg = compare(got, exp, what)
    print(msg)
    assert ok, msg
    return out


def test_forward_tiny():
    d = make_moe_case(CONFIGS["tiny"], seed=0, device=DEV)
    _run_parity(d, what="tiny")


@pytest.mark.parametrize("tuned", [False, True], ids=["built_in", "tuned_table"])
def test_forward_decode(tuned):
    # the tuned table is the launch configuration bench.py times (32-token
    # tiles, both projections in one launch)
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    binding.moelora_load_tuning(table if tuned else None)
    try:
        d = make_moe_case(CONFIGS["decode"], seed=0, device=DEV)
        _run_parity(d, what=f"decode ({'tuned' if tuned else 'built-in'})", key="decode")
    finally:
        binding.moelora_load_tuning(None)


@pytest.mark.parametrize("tuned", [False, True], ids=["built_in", "tuned_table"])
def test_forward_prefill_full(tuned):
    # all 4096 tokens (16384 routed pairs on 2-SM tiles) against the oracle
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    binding.moelora_load_tuning(table if tuned else None)
    try:
        d = make_moe_case(CONFIGS["prefill"], seed=0, device=DEV)
        _run_parity(d, what=f"prefill (all 4096 tokens, {'tuned' if tuned else 'built-in'})",
                    key="prefill")
    finally:
        binding.moelora_load_tuning(None)


@pytest.mark.parametrize("tuned", [False, True], ids=["built_in", "tuned_table"])
def test_forward_skewed_full(tuned):
    # the tuned table (the launch configuration bench.py times) runs this
    # workload on larger token tiles than the built-in choice; all 256 tokens
    # (1536 routed pairs over the Zipf-loaded experts) against the oracle
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    binding.moelora_load_tuning(table if tuned else None)
    try:
        d = make_moe_case(CONFIGS["skewed"], seed=0, device=DEV)
        _run_parity(d, what=f"skewed (all 256 tokens, {'tuned' if tuned else 'built-in'})",
                    key="skewed")
    finally:
        binding.moelora_load_tuning(None)


SMALL = [
    # T, H, I, E, k, L, r
    (1, 64, 64, 1, 1, 1, 16),
    (5, 136, 72, 3, 2, 2, 16),       # H % 128 != 0, I % 64 != 0
    (33, 256, 192, 4, 4, 3, 32),     # k == E
    (70, 128, 128, 6, 2, 5, 64),
    (19, 192, 320, 5, 3, 2, 128),
    (40, 200, 136, 7, 2, 0, 0),      # no LoRA
    (300, 264, 264, 8, 2, 4, 16),    # several tiles per expert, ragged tail
    (8, 136, 2048, 4, 2, 2, 16),     # few rows per expert, long K: the down phase splits K
    (600, 256, 200, 2, 1, 3, 32),    # 256-row tiles on CTA pairs, partial tiles and feature blocks
    (520, 136, 72, 2, 2, 2, 128),    # CTA pairs, rank 128: one adapter per CTA in a shrink item
    (37, 200, 264, 5, 2, 3, 48),     # rank 48: 16-wide expand chunks, two adapters per shrink tile
    (530, 136, 200, 2, 2, 3, 48),    # CTA pairs at rank 48: two adapters on each CTA of an item
    (23, 264, 136, 4, 3, 2, 96),     # rank 96: 32-wide chunks, one adapter per shrink tile
    (300, 128, 256, 2, 1, 3, 80),    # CTA pairs at rank 80
    (45, 256, 128, 3, 2, 2, 112),    # rank 112
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"T{s[0]}_H{s[1]}_I{s[2]}_E{s[3]}_k{s[4]}_L{s[5]}_r{s[6]}" for s in SMALL])
def test_forward_small_shapes(shape):
    T, H, I, E, k, L, r = shape
    c = small_moe_case(T, H, I, E, k, L, r, adapters="uniform_with_none" if L else "uniform")
    if L == 0:
        c = small_moe_case(T, H, I, E, k, 1, 16)
    d = make_moe_case(c, seed=11, device=DEV, lora=L > 0)
    if L == 0:
        d["lora_ids"] = torch.full((T,), -1, dtype=torch.int32, device=DEV)
    _run_parity(d, what=str(shape))


def _random_shapes(n, seed):
    """Seeded random small layer shapes: sizes off the tile grid, any rank the
    library takes, both routings and adapter mixes, with or without LoRA."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.integers(1, 17))
        k = int(rng.integers(1, min(E, 8) + 1))
        L = int(rng.integers(0, 6))
        out.append(dict(T=int(rng.integers(1, 301)), H=8 * int(rng.integers(8, 41)),
                        I=8 * int(rng.integers(8, 41)), E=E, k=k, L=L,
                        r=16 * int(rng.integers(1, 9)) if L else 0,
                        routing=str(rng.choice(["uniform", "zipf"])),
                        adapters=str(rng.choice(["uniform_with_none", "zipf"]))))
    return out


SPLIT_SHAPES = [SMALL[4], SMALL[6], SMALL[8], SMALL[9], SMALL[11], SMALL[13]]


@pytest.mark.parametrize("splits", [2, 3, 5])
@pytest.mark.parametrize("shape", SPLIT_SHAPES,
                         ids=[f"T{s[0]}_H{s[1]}_I{s[2]}_E{s[3]}_k{s[4]}_L{s[5]}_r{s[6]}" for s in SPLIT_SHAPES])
def test_forward_shrink_split_k(monkeypatch, shape, splits):
    """Shrink items cut into K splits (forced; the built-in choice splits
    only long reductions on single-CTA tiles): each split's fp32 part is
    summed in split order by the last split to finish, on single CTAs and
    CTA pairs, with the gate_up hi/lo z and every tested rank."""
    monkeypatch.setenv("MOELORA_SHRINK_SPLITS", str(splits))
    T, H, I, E, k, L, r = shape
    d = make_moe_case(small_moe_case(T, H, I, E, k, L, r), seed=21, device=DEV)
    out = _run_parity(d, what=f"{shape} shrink splits {splits}")
    again = _gpu_forward(d)
    assert torch.equal(out, again)          # the order of arrival does not matter


# H >= 48 K blocks so that three splits keep at least 16 K blocks each
GU_SPLIT_SHAPES = [(8, 3072, 2048, 1, 1, 4, 16), (40, 3072, 1024, 3, 2, 3, 32), (70, 3200, 520, 2, 2, 2, 64)]


@pytest.mark.parametrize("two_phase", ["0", "1"])
@pytest.mark.parametrize("splits", [2, 3])
@pytest.mark.parametrize("shape", GU_SPLIT_SHAPES,
                         ids=[f"T{s[0]}_H{s[1]}_I{s[2]}_E{s[3]}_k{s[4]}_L{s[5]}_r{s[6]}" for s in GU_SPLIT_SHAPES])
def test_forward_gate_up_split_k(monkeypatch, shape, splits, two_phase):
    """The gate_up phase cut into K splits (forced): each split's fp32 part
    is summed in split order by the last split to arrive, which applies
    SiLU(gate) * up; with one launch per projection and with both in one
    launch (whose down items then wait for one count per weight tile)."""
    T, H, I, E, k, L, r = shape
    d = make_moe_case(small_moe_case(T, H, I, E, k, L, r), seed=31, device=DEV)
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
    unsplit = binding.moelora_workspace_bytes(dims)
    monkeypatch.setenv("MOELORA_GU_KSPLIT", str(splits))
    monkeypatch.setenv("MOELORA_TWO_PHASE", two_phase)
    assert binding.moelora_workspace_bytes(dims) > unsplit   # the split's parts are planned
    out = _run_parity(d, what=f"{shape} gate_up splits {splits}")
    again = _gpu_forward(d)
    assert torch.equal(out, again)          # the order of arrival does not matter


# CTA-pair shapes for the spread shrink order: ragged tiles, several per
# expert, tiles with more adapters than one shrink item stacks and tiles
# with none (adapter -1), every rank
SPREAD_SHAPES = [(700, 512, 384, 3, 2, 6, 16), (520, 256, 512, 5, 3, 9, 32), (300, 384, 256, 2, 1, 3, 64),
                 (900, 192, 320, 7, 2, 12, 48)]


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("shape", SPREAD_SHAPES,
                         ids=[f"T{s[0]}_H{s[1]}_I{s[2]}_E{s[3]}_k{s[4]}_L{s[5]}_r{s[6]}" for s in SPREAD_SHAPES])
def test_forward_spread_shrink_order(monkeypatch, shape, splits):
    """CTA-pair launches with the shrink entries spread over the first K
    split (forced here; the built-in choice spreads them only when the token
    rows are more than L2 keeps): each tile's shrink slots, empty ones
    included, a wave of items ahead of its main items.  Compared with the
    oracle, and bit for bit with the all-first order: the claim order
    changes no sum."""
    monkeypatch.setenv("MOELORA_TN", "256")
    monkeypatch.setenv("MOELORA_SHRINK_SPLITS", str(splits))
    T, H, I, E, k, L, r = shape
    d = make_moe_case(small_moe_case(T, H, I, E, k, L, r), seed=41, device=DEV)
    monkeypatch.setenv("MOELORA_SPREAD_SHRINK", "1")
    out = _run_parity(d, what=f"{shape} spread shrink, {splits} shrink splits")
    monkeypatch.setenv("MOELORA_SPREAD_SHRINK", "0")
    assert torch.equal(out, _gpu_forward(d))


@pytest.mark.parametrize("spread", ["0", "1"])
def test_linear_spread_shrink_order(monkeypatch, spread):
    """The dense linear on CTA pairs with its shrink entries spread over the
    first K split and all first: the same bits, and the oracle's result."""
    monkeypatch.setenv("MOELORA_TN", "256")
    monkeypatch.setenv("MOELORA_SPREAD_SHRINK", spread)
    g = torch.Generator(device=DEV).manual_seed(43)
    T, K, N, L, r = 777, 512, 640, 9, 16
    x = torch.randn(T, K, generator=g, device=DEV).bfloat16()
    W = (torch.randn(N, K, generator=g, device=DEV) * K ** -0.5).bfloat16()
    A = (torch.randn(L, r, K, generator=g, device=DEV) * K ** -0.5).bfloat16()
    B = (torch.randn(L, N, r, generator=g, device=DEV) * r ** -0.5).bfloat16()
    lo = torch.randint(-1, L, (T,), generator=g, device=DEV).int()
    out = binding.moe_lora_linear(x, lo, W, A, B)
    n = np_inputs({"x": x, "W": W, "A": A, "B": B})
    exp = ref.moe_lora_linear_ref(n["x"], lo.cpu().numpy(), n["W"], n["A"], n["B"])
    ok, msg = compare(out, exp, f"linear spread={spread}")
    print(msg)
    assert ok, msg
    monkeypatch.setenv("MOELORA_SPREAD_SHRINK", "1" if spread == "0" else "0")
    assert torch.equal(out, binding.moe_lora_linear(x, lo, W, A, B))


@pytest.mark.parametrize("name", ["decode", "dense_mlp_t1", "tiny"])
def test_align_weight_prefetch_changes_no_bit(monkeypatch, name):
    """The small align's L2 weight prefetch (whole experts for the decode
    batch, the first K split's row slices for the dense MLP at T = 1) only
    moves lines into L2: the output is the same bits with it off, and the
    batch still matches the oracle."""
    c = CONFIGS[name]
    d = make_moe_case(c, seed=0, device=DEV)
    out = _gpu_forward(d).clone()
    monkeypatch.setenv("MOELORA_PF_MB", "0")
    assert torch.equal(out, _gpu_forward(d))
    monkeypatch.setenv("MOELORA_PF_MB", "64")      # a larger prefetch, still no effect on the bits
    assert torch.equal(out, _gpu_forward(d))
    if name == "tiny":
        n = np_inputs(d)
        ok, msg = compare(out, _oracle_forward(n), f"{name} with the prefetch")
        assert ok, msg


def test_linear_weight_prefetch_changes_no_bit(monkeypatch):
    """The dense linear's align prefetch (row slices of the first K split):
    the same bits with it off."""
    d = make_linear_case(CONFIGS["dense_t1"], seed=0, device=DEV)
    out = binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"]).clone()
    monkeypatch.setenv("MOELORA_PF_MB", "0")
    assert torch.equal(out, binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"]))


@pytest.mark.parametrize("shape", _random_shapes(24, 17), ids=lambda s: "T{T}_H{H}_I{I}_E{E}_k{k}_L{L}_r{r}".format(**s))
def test_forward_random_shapes(shape):
    s = shape
    L, r = (s["L"], s["r"]) if s["L"] else (1, 16)
    c = small_moe_case(s["T"], s["H"], s["I"], s["E"], s["k"], L, r, adapters=s["adapters"],
                       routing=s["routing"])
    d = make_moe_case(c, seed=23, device=DEV, lora=s["L"] > 0)
    if s["L"] == 0:
        d["lora_ids"] = torch.full((s["T"],), -1, dtype=torch.int32, device=DEV)
    _run_parity(d, what=str(s))


def test_forward_many_experts_top8():
    # A stress shape beyond the five workloads: gate-weighted sums of eight
    # Zipf-routed pairs put some outputs at 9-10 x RMS, where one bf16 ulp
    # of the output is 2-4 x the max-abs bound's 3e-2 x RMS; with the
    # activation rounded to bf16 as the down GEMM's operand, a float64
    # emulation of the kernel's rounding points already exceeds the bound at
    # 1-3 of the 131k elements on 2 of 3 seeds.  Compared on 64 sampled
    # tokens; the five workloads are compared over their whole batches.
    c = small_moe_case(1024, 128, 192, 64, 8, 4, 16, adapters="zipf", routing="zipf")
    d = make_moe_case(c, seed=6, device=DEV)
    rng = np.random.default_rng(3)
    _run_parity(d, tokens=np.sort(rng.choice(1024, size=64, replace=False)), what="E64 top-8")


def test_forward_maximum_bins_and_top32():
    """The largest expert x adapter table (E = 1024, L = 10: 11264 bins) and
    the largest top-k the router kernel takes (k = 32)."""
    # (compared on sampled tokens for the reason given in the top-8 test: a
    # Zipf-routed output at 8.6 x RMS sits one bf16 half-ulp from the bound)
    c = small_moe_case(1500, 64, 128, 1024, 4, 10, 16, routing="zipf")
    d = make_moe_case(c, seed=12, device=DEV)
    rng = np.random.default_rng(12)
    _run_parity(d, tokens=np.sort(rng.choice(1500, size=48, replace=False)), what="E1024 L10")
    c = small_moe_case(96, 128, 64, 64, 32, 3, 32)
    d = make_moe_case(c, seed=13, device=DEV)
    _run_parity(d, what="top-32")


def test_forward_duplicate_experts_in_topk():
    """A token may name the same expert more than once in its top-k: each
    entry is its own routed pair (same expert and adapter, its own gate
    weight), so the output counts the expert once per entry."""
    c = small_moe_case(50, 128, 64, 4, 3, 2, 16)
    d = make_moe_case(c, seed=14, device=DEV)
    g = torch.Generator().manual_seed(14)
    ids = torch.randint(0, 4, (50, 3), generator=g, dtype=torch.int32)
    ids[:10, 1] = ids[:10, 0]              # a pair of equal entries
    ids[10:15, :] = ids[10:15, :1]         # all three entries equal
    d["topk_ids"] = ids.to(DEV)
    _check_align(ids, d["lora_ids"].cpu(), 4, 2, 16)
    _run_parity(d, what="duplicate experts")


def test_forward_empty_batch():
    c = small_moe_case(4, 64, 64, 4, 2, 2, 16)
    d = make_moe_case(c, seed=0, device=DEV)
    e = {k: (v[:0] if k in ("x", "topk_ids", "topk_weights", "lora_ids") else v) for k, v in d.items()}
    out = _gpu_forward(e)
    torch.cuda.synchronize()
    assert out.shape == (0, 64)


def test_forward_all_one_expert_and_no_adapter():
    c = small_moe_case(200, 128, 128, 4, 1, 3, 32)
    d = make_moe_case(c, seed=5, device=DEV)
    d["topk_ids"] = torch.full((200, 1), 3, dtype=torch.int32, device=DEV)
    d["topk_weights"] = torch.ones((200, 1), dtype=torch.float32, device=DEV)
    _run_parity(d, what="one expert")
    d["lora_ids"] = torch.full((200,), -1, dtype=torch.int32, device=DEV)
    _run_parity(d, what="one expert, no adapters")


@pytest.mark.parametrize("name", ["tiny", "decode", "dense_mlp_t8"])
def test_forward_deterministic_and_graph_capturable(name):
    """Two eager calls are bit-identical; a captured call replays to the same
    output; after the routing, adapters and activations are changed in place,
    a second replay equals an eager call on the new inputs (nothing that
    depends on the data is baked into the graph).  decode and the dense MLP
    run split shrink items and K-split down phases inside the graph."""
    d = make_moe_case(CONFIGS[name], seed=2, device=DEV)
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
    ws = binding.alloc_workspace(binding.moelora_workspace_bytes(dims))
    a = _gpu_forward(d, ws=ws).clone()
    b = _gpu_forward(d, ws=ws).clone()
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _gpu_forward(d, ws=ws, out=out)       # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        _gpu_forward(d, ws=ws, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, a)
    # new inputs in the captured buffers
    d2 = make_moe_case(CONFIGS[name], seed=5, device=DEV)
    for k in ("x", "topk_ids", "topk_weights", "lora_ids"):
        d[k].copy_(d2[k])
    g.replay()
    torch.cuda.synchronize()
    ws2 = binding.alloc_workspace(binding.moelora_workspace_bytes(dims))
    assert torch.equal(out, _gpu_forward(d, ws=ws2))


def test_linear_graph_replay_with_new_inputs():
    c = CONFIGS["dense_t64"]
    d = make_linear_case(c, seed=1, device=DEV)
    dims = binding.moelora_linear_dims(c.T, c.K, c.N, c.L, c.r)
    ws = binding.alloc_workspace(binding.moelora_linear_workspace_bytes(dims))
    out = torch.empty((c.T, c.N), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"], out=out, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"], out=out, ws=ws)
    d2 = make_linear_case(c, seed=2, device=DEV)
    d["x"].copy_(d2["x"])
    d["lora_ids"].copy_(d2["lora_ids"])
    g.replay()
    torch.cuda.synchronize()
    eager = binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"])
    assert torch.equal(out, eager)


@pytest.mark.parametrize("name", ["decode", "tiny", "dense_mlp_t64"])
def test_two_phase_launch_equals_two_launches(monkeypatch, name):
    """Both projections in one persistent launch (single-CTA tiles) give the
    same bits as one launch per projection: the items and their arithmetic
    are the same, only the order in which CTAs take them differs."""
    d = make_moe_case(CONFIGS[name], seed=3, device=DEV)
    outs, names = {}, {}
    for ph in ("1", "2"):
        monkeypatch.setenv("MOELORA_TWO_PHASE", "0" if ph == "1" else "1")
        outs[ph] = _gpu_forward(d).clone()
        names[ph] = binding.moelora_last_launches()
    assert "gemm_gate_up_down" in names["2"] and "gemm_gate_up_down" not in names["1"], names
    assert torch.equal(outs["1"], outs["2"])
    n = np_inputs(d, lazy=True)
    ok, msg = compare(outs["2"], _oracle_forward(n), name)
    assert ok, msg


def test_back_to_back_calls_on_one_stream():
    # Calls of different shapes (small-batch path with the fused row gather,
    # the multi-kernel align path, the dense linear) queued on one stream
    # without a synchronisation in between, some sharing a workspace: every
    # launch may begin before its predecessor ends, so each result must still
    # equal the same call made alone.
    small = make_moe_case(CONFIGS["tiny"], seed=3, device=DEV)
    big_c = small_moe_case(1100, 128, 192, 8, 2, 3, 32)   # > 1024 entries: hist/scan/scatter align
    big = make_moe_case(big_c, seed=4, device=DEV)
    lin_c = CONFIGS["dense_t8"]
    lin = make_linear_case(lin_c, seed=5, device=DEV)

    def ws_for(d):
        dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
        return binding.alloc_workspace(binding.moelora_workspace_bytes(dims))

    ws_small, ws_big = ws_for(small), ws_for(big)
    alone = {}
    alone["small"] = _gpu_forward(small, ws=ws_small).clone()
    alone["big"] = _gpu_forward(big, ws=ws_big).clone()
    alone["lin"] = binding.moe_lora_linear(lin["x"], lin["lora_ids"], lin["W"], lin["A"], lin["B"]).clone()
    torch.cuda.synchronize()

    small2 = dict(small, lora_ids=torch.roll(small["lora_ids"], 1))   # other routing, same workspace
    outs = []
    for _ in range(3):
        outs.append(("small", _gpu_forward(small, ws=ws_small)))
        outs.append(("big", _gpu_forward(big, ws=ws_big)))
        outs.append(("small2", _gpu_forward(small2, ws=ws_small)))
        outs.append(("lin", binding.moe_lora_linear(lin["x"], lin["lora_ids"], lin["W"], lin["A"], lin["B"])))
    torch.cuda.synchronize()
    alone["small2"] = _gpu_forward(small2, ws=ws_small).clone()
    torch.cuda.synchronize()
    for name, out in outs:
        assert torch.equal(out, alone[name]), name


def test_forward_bad_index_flag():
    d = make_moe_case(CONFIGS["tiny"], seed=0, device=DEV)
    dims = binding.dims_of(d["x"], d["topk_ids"], d["W_gate_up"], d["W_down"], d["A_gu"])
    ws = binding.alloc_workspace(binding.moelora_workspace_bytes(dims))
    _gpu_forward(d, ws=ws)
    assert binding.moelora_get_error(ws) == 0
    bad = dict(d, lora_ids=d["lora_ids"].clone())
    bad["lora_ids"][5] = 9
    _gpu_forward(bad, ws=ws)
    assert binding.moelora_get_error(ws) == -6
    _gpu_forward(d, ws=ws)
    assert binding.moelora_get_error(ws) == 0


# ------------------------------------------------------------------ dense linear
@pytest.mark.parametrize("tuned", [False, True], ids=["built_in", "tuned_table"])
@pytest.mark.parametrize("T", DENSE_T_SWEEP)
def test_linear_dense(T, tuned):
    # the tuned table is the launch configuration bench.py times (its token
    # tile and K split differ from the built-in choice for some T)
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    c = CONFIGS[f"dense_t{T}"]
    d = make_linear_case(c, seed=0, device=DEV)
    binding.moelora_load_tuning(table if tuned else None)
    try:
        out = binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"])
        torch.cuda.synchronize()
    finally:
        binding.moelora_load_tuning(None)
    # every token of the batch against the oracle
    key = f"dense_t{T}"
    if key not in _ORACLE:
        n = np_inputs({k: d[k] for k in ("x", "W", "A", "B")})
        _ORACLE[key] = ref.moe_lora_linear_ref(n["x"], d["lora_ids"].cpu().numpy(), n["W"], n["A"],
                                               n["B"])
    ok, msg = compare(out, _ORACLE[key], f"dense T={T} ({'tuned' if tuned else 'built-in'})")
    print(msg)
    assert ok, msg


@pytest.mark.parametrize("tuned", [False, True], ids=["built_in", "tuned_table"])
@pytest.mark.parametrize("T", DENSE_T_SWEEP)
def test_forward_dense_mlp(T, tuned):
    """The whole layer at E = 1, top-1 (a dense two-projection MLP with
    per-token LoRA) with the dense shapes H = 8192, I = 14336."""
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    d = make_moe_case(CONFIGS[f"dense_mlp_t{T}"], seed=0, device=DEV)
    binding.moelora_load_tuning(table if tuned else None)
    try:
        _run_parity(d, what=f"dense MLP T={T} ({'tuned' if tuned else 'built-in'})",
                    key=f"dense_mlp_t{T}")
    finally:
        binding.moelora_load_tuning(None)


@pytest.mark.parametrize("T", [12, 100, 700])
def test_forward_off_ladder_batch_sizes_under_the_tuned_table(T):
    """Batch sizes that the tuning sweep did not sample take the choice of
    their batch-size bucket in the shipped table; compared in full."""
    import dataclasses
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    base = CONFIGS["prefill"] if T >= 512 else CONFIGS["decode"]
    c = dataclasses.replace(base, name=f"decode_shapes_t{T}", T=T)
    d = make_moe_case(c, seed=4, device=DEV)
    binding.moelora_load_tuning(table)
    try:
        _run_parity(d, what=f"decode shapes T={T} (tuned bucket)")
    finally:
        binding.moelora_load_tuning(None)


@pytest.mark.parametrize("T", [3, 24, 200])
def test_linear_off_ladder_batch_sizes_under_the_tuned_table(T):
    import dataclasses
    import os
    table = os.path.join(os.path.dirname(binding.__file__), "tuning")
    c = dataclasses.replace(CONFIGS["dense_t1"], name=f"dense_t{T}", T=T)
    d = make_linear_case(c, seed=4, device=DEV)
    binding.moelora_load_tuning(table)
    try:
        out = binding.moe_lora_linear(d["x"], d["lora_ids"], d["W"], d["A"], d["B"])
        torch.cuda.synchronize()
    finally:
        binding.moelora_load_tuning(None)
    n = np_inputs({k: d[k] for k in ("x", "W", "A", "B")})
    exp = ref.moe_lora_linear_ref(n["x"], d["lora_ids"].cpu().numpy(), n["W"], n["A"], n["B"])
    ok, msg = compare(out, exp, f"dense T={T} (tuned bucket)")
    print(msg)
    assert ok, msg


@pytest.mark.parametrize("seed", range(12))
def test_linear_random_shapes(seed):
    # seeded random dense multi-LoRA linears: ragged T, K and N off the tile
    # grid, any rank the library takes, some tokens without an adapter
    rng = np.random.default_rng(100 + seed)
    T, K, N = int(rng.integers(1, 600)), 8 * int(rng.integers(8, 80)), 8 * int(rng.integers(8, 80))
    L = int(rng.integers(0, 9))
    r = 16 * int(rng.integers(1, 9)) if L else 0
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(T, K, generator=g, device=DEV).bfloat16()
    W = (torch.randn(N, K, generator=g, device=DEV) * K ** -0.5).bfloat16()
    A = (torch.randn(L, r, K, generator=g, device=DEV) * K ** -0.5).bfloat16() if L else None
    B = (torch.randn(L, N, r, generator=g, device=DEV) * r ** -0.5).bfloat16() if L else None
    lo = (torch.randint(-1, L, (T,), generator=g, device=DEV) if L else torch.full((T,), -1, device=DEV)).int()
    out = binding.moe_lora_linear(x, lo, W, A, B)
    n = np_inputs({"x": x, "W": W, **({"A": A, "B": B} if L else {})})
    exp = ref.moe_lora_linear_ref(n["x"], lo.cpu().numpy(), n["W"], n.get("A"), n.get("B"))
    ok, msg = compare(out, exp, f"linear T={T} K={K} N={N} L={L} r={r}")
    assert ok, msg


def test_linear_small_no_lora_and_ragged():
    g = torch.Generator(device=DEV).manual_seed(4)
    for (T, K, N, L, r) in [(3, 64, 136, 0, 0), (45, 200, 264, 3, 32), (260, 128, 128, 2, 64),
                            (33, 192, 264, 3, 48), (270, 136, 128, 2, 96)]:
        x = torch.randn(T, K, generator=g, device=DEV).bfloat16()
        W = (torch.randn(N, K, generator=g, device=DEV) * K ** -0.5).bfloat16()
        A = (torch.randn(L, r, K, generator=g, device=DEV) * K ** -0.5).bfloat16() if L else None
        B = (torch.randn(L, N, r, generator=g, device=DEV) * r ** -0.5).bfloat16() if L else None
        lo = (torch.randint(-1, L, (T,), generator=g, device=DEV) if L else torch.full((T,), -1, device=DEV)).int()
        out = binding.moe_lora_linear(x, lo, W, A, B)
        n = np_inputs({"x": x, "W": W, **({"A": A, "B": B} if L else {})})
        exp = ref.moe_lora_linear_ref(n["x"], lo.cpu().numpy(), n["W"], n.get("A"), n.get("B"))
        ok, msg = compare(out, exp, f"linear {(T, K, N, L, r)}")
        assert ok, msg


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("T,E,k", [(16, 32, 4), (300, 64, 6), (5, 1024, 8), (64, 8, 8), (7, 3, 1)])
def test_route_matches_oracle(T, E, k):
    g = torch.Generator().manual_seed(T * 131 + E)
    logits = torch.randn(T, E, generator=g)
    logits[0, :min(E, 4)] = 0.25            # ties: the lower index wins
    ids, w = binding.moe_lora_route(logits.to(DEV), k)
    torch.cuda.synchronize()
    eids, ew = ref.router_topk_ref(logits.numpy(), k)
    assert np.array_equal(ids.cpu().numpy(), eids)
    assert np.abs(w.cpu().numpy() - ew).max() < 2e-6


def _logits_for(d, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(d["x"].shape[0], E, generator=g).to(DEV)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_forward_routed_equals_route_then_forward(name):
    c = CONFIGS[name]
    d = make_moe_case(c, seed=0, device=DEV)
    logits = _logits_for(d, c.E, 5)
    out_r = binding.moe_lora_forward_routed(d["x"], logits, c.k, d["lora_ids"], d["W_gate_up"],
                                            d["W_down"], d["A_gu"], d["B_gu"], d["A_d"], d["B_d"])
    ids, w = binding.moe_lora_route(logits, c.k)
    out_s = binding.moe_lora_forward(d["x"], ids, w, d["lora_ids"], d["W_gate_up"], d["W_down"],
                                     d["A_gu"], d["B_gu"], d["A_d"], d["B_d"])
    torch.cuda.synchronize()
    assert torch.equal(out_r, out_s)
    # and against the oracle with the oracle's own routing
    eids, ew = ref.router_topk_ref(logits.cpu().numpy(), c.k)
    assert np.array_equal(ids.cpu().numpy(), eids)
    n = np_inputs(d)
    exp = ref.moe_lora_forward_ref(n["x"], eids, ew, n["lora_ids"], n["W_gate_up"], n["W_down"],
                                   n["A_gu"], n["B_gu"], n["A_d"], n["B_d"])
    ok, msg = compare(out_r, exp, f"routed {name}")
    assert ok, msg


def test_forward_routed_large_batch():
    # above the single-CTA align: router kernel, then the three align kernels
    c = small_moe_case(600, 128, 128, 16, 4, 3, 16)
    d = make_moe_case(c, seed=2, device=DEV)
    logits = _logits_for(d, c.E, 8)
    out_r = binding.moe_lora_forward_routed(d["x"], logits, c.k, d["lora_ids"], d["W_gate_up"],
                                            d["W_down"], d["A_gu"], d["B_gu"], d["A_d"], d["B_d"])
    ids, w = binding.moe_lora_route(logits, c.k)
    out_s = binding.moe_lora_forward(d["x"], ids, w, d["lora_ids"], d["W_gate_up"], d["W_down"],
                                     d["A_gu"], d["B_gu"], d["A_d"], d["B_d"])
    torch.cuda.synchronize()
    assert torch.equal(out_r, out_s)


# ------------------------------------------------------------------ merged-weight fast path
@pytest.mark.parametrize("shape", [(4, 136, 72, 3, 16), (2, 256, 512, 4, 64), (1, 264, 200, 2, 128),
                                   (3, 200, 136, 2, 48), (2, 1000, 712, 2, 96), (5, 128, 1224, 3, 32),
                                   (2, 392, 264, 2, 80), (1, 136, 520, 1, 112)])
def test_merge_adapter_weights(shape):
    # ragged rows and columns (partial 128 x 128 tiles), several row ranges
    # per column block, every chunk width of the rank (16, 32, 64)
    E, H, I, L, r = shape
    c = small_moe_case(8, H, I, E, 1, L, r)
    d = make_moe_case(c, seed=3, device=DEV)
    a = L - 1
    Wgu, Wd = binding.moe_lora_merge_adapter(a, d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"],
                                             d["A_d"], d["B_d"])
    torch.cuda.synchronize()
    n = np_inputs(d)
    exp_gu = ref.as_f64(n["W_gate_up"]) + np.einsum("ecq,eqh->ech", ref.as_f64(n["B_gu"][a]),
                                                    ref.as_f64(n["A_gu"][a]))
    exp_d = ref.as_f64(n["W_down"]) + np.einsum("ehq,eqi->ehi", ref.as_f64(n["B_d"][a]),
                                                ref.as_f64(n["A_d"][a]))
    for got, exp in ((Wgu, exp_gu), (Wd, exp_d)):
        g = got.float().cpu().numpy().astype(np.float64)
        # one bf16 rounding of the fp32 sum: within 2^-8 relative (+ a tiny absolute floor)
        assert np.all(np.abs(g - exp) <= 2.0 ** -8 * np.abs(exp) + 1e-6)


@pytest.mark.parametrize("name", ["decode", "skewed"])
def test_merge_adapter_weights_full_size(name):
    """The merge at the bench workloads' layer sizes, every merged element of
    a sample of experts against float64 W + B A (one bf16 rounding)."""
    c = CONFIGS[name]
    d = make_moe_case(c, seed=0, device=DEV)
    a = c.L - 1
    Wgu, Wd = binding.moe_lora_merge_adapter(a, d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"],
                                             d["A_d"], d["B_d"])
    torch.cuda.synchronize()
    from lora_mixture_experts_gb300.inputs import bf16_bits
    for e in (0, c.E // 2 + 1, c.E - 1):
        for W, B, A, got in ((d["W_gate_up"], d["B_gu"], d["A_gu"], Wgu), (d["W_down"], d["B_d"], d["A_d"], Wd)):
            exact = ref.as_f64(bf16_bits(W[e])) + ref.as_f64(bf16_bits(B[a, e])) @ ref.as_f64(bf16_bits(A[a, e]))
            g = ref.as_f64(bf16_bits(got[e]))
            assert np.all(np.abs(g - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-6), (name, e)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_merged_fast_path_matches_lora_layer(name):
    c = CONFIGS[name]
    d = make_moe_case(c, seed=1, device=DEV)
    a = 2
    d["lora_ids"] = torch.full((c.T,), a, dtype=torch.int32, device=DEV)   # one adapter for the batch
    Wgu, Wd = binding.moe_lora_merge_adapter(a, d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"],
                                             d["A_d"], d["B_d"])
    no_lora = torch.full((c.T,), -1, dtype=torch.int32, device=DEV)
    out = binding.moe_lora_forward(d["x"], d["topk_ids"], d["topk_weights"], no_lora, Wgu, Wd)
    torch.cuda.synchronize()
    n = np_inputs(d)
    exp = _oracle_forward(n)                # the LoRA layer, every token on adapter a
    ok, msg = compare(out, exp, f"merged {name}")
    assert ok, msg
