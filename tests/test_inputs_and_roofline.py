"""Host-side checks of the seeded workload generator (shapes, reproducibility,
the distributions the workloads state) and of the algorithmic byte / FLOP
accounting the benchmark's roofline uses (against a brute-force count)."""
import numpy as np
import pytest
import torch

from lora_mixture_experts_gb300 import inputs, roofline
from lora_mixture_experts_gb300.inputs import CONFIGS, make_moe_case, make_routing, small_moe_case


def test_routing_shapes_and_renormalisation():
    for name in ("tiny", "decode", "prefill", "skewed"):
        c = CONFIGS[name]
        ids, w, lo = make_routing(c, seed=0)
        assert ids.shape == (c.T, c.k) and ids.dtype == torch.int32
        assert w.shape == (c.T, c.k) and w.dtype == torch.float32
        assert lo.shape == (c.T,) and lo.dtype == torch.int32
        assert int(ids.min()) >= 0 and int(ids.max()) < c.E
        assert int(lo.min()) >= -1 and int(lo.max()) < c.L
        # distinct experts per token, weights renormalised and descending
        assert all(len(set(r.tolist())) == c.k for r in ids)
        assert torch.allclose(w.sum(1), torch.ones(c.T), atol=1e-6)
        assert bool((w[:, :-1] >= w[:, 1:]).all())


def test_routing_reproducible_and_seed_dependent():
    c = CONFIGS["decode"]
    a = make_routing(c, seed=3)
    b = make_routing(c, seed=3)
    d = make_routing(c, seed=4)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], d[0])


def test_adapter_recipes():
    _, _, lo = make_routing(CONFIGS["prefill"], seed=0)
    assert torch.equal(lo, (torch.arange(4096) // 512).int())          # one adapter per request
    _, _, lo = make_routing(CONFIGS["tiny"], seed=0)
    assert set(lo.tolist()) <= {-1, 0, 1, 2, 3} and (lo == -1).any()
    _, _, lo = make_routing(CONFIGS["decode"], seed=0)
    assert int(lo.min()) >= 0                                            # every token has an adapter


def test_skewed_routing_follows_zipf():
    c = CONFIGS["skewed"]
    ids, _, lo = make_routing(c, seed=0)
    load = np.bincount(ids.numpy().ravel(), minlength=c.E)
    # expert 0 is the most loaded and load falls with the expert index
    assert load[0] == load.max()
    assert load[:8].sum() > load[32:].sum()
    none = float((lo == -1).float().mean())
    assert 0.03 < none < 0.2                                            # ~10% without adapter
    a = lo[lo >= 0].numpy()
    assert np.bincount(a, minlength=c.L)[0] == np.bincount(a, minlength=c.L).max()


def test_weight_scales():
    c = small_moe_case(32, 512, 256, 4, 2, 2, 16)
    d = make_moe_case(c, seed=1)
    def std(t):
        return float(t.float().std())
    assert abs(std(d["x"]) - 1.0) < 0.05
    assert abs(std(d["W_gate_up"]) - 512 ** -0.5) < 0.1 * 512 ** -0.5   # fan-in H
    assert abs(std(d["W_down"]) - 256 ** -0.5) < 0.1 * 256 ** -0.5      # fan-in I
    assert abs(std(d["A_gu"]) - 512 ** -0.5) < 0.1 * 512 ** -0.5
    assert abs(std(d["B_gu"]) - 16 ** -0.5) < 0.1 * 16 ** -0.5
    assert abs(std(d["A_d"]) - 256 ** -0.5) < 0.1 * 256 ** -0.5
    assert all(d[k].dtype == torch.bfloat16 for k in ("x", "W_gate_up", "W_down", "A_gu", "B_gu", "A_d", "B_d"))


def _brute_work(ids, lo, H, I, r):
    T, k = ids.shape
    experts, ea, lora_pairs = set(), set(), 0
    for t in range(T):
        for j in range(k):
            experts.add(int(ids[t, j]))
            if lo[t] >= 0:
                ea.add((int(ids[t, j]), int(lo[t])))
                lora_pairs += 1
    b = len(experts) * 3 * I * H * 2 + len(ea) * (H * r + r * 2 * I + I * r + r * H) * 2 \
        + 2 * T * H * 2 + T * k * 8 + T * 4
    f = T * k * 2 * (2 * I * H + I * H) + lora_pairs * 2 * (H * r + r * 2 * I + I * r + r * H)
    return b, f


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_roofline_counts_match_brute_force(name):
    c = CONFIGS[name]
    ids, _, lo = make_routing(c, seed=0)
    layer, gu, dn = roofline.moe_layer_work(ids.numpy(), lo.numpy(), c.H, c.I, c.r)
    b, f = _brute_work(ids.numpy(), lo.numpy(), c.H, c.I, c.r)
    assert layer.bytes == b and layer.flops == f
    assert gu.flops + dn.flops == f


def test_roofline_time_and_bound():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 50.0, "source": "t"}
    w = roofline.Work(bytes=1e9, flops=1e12)
    assert roofline.roofline_time_s(w, peaks) == pytest.approx(1e-2)           # tensor: 1e12/1e14
    assert roofline.roofline_time_s(w, peaks, sustained=True) == pytest.approx(2e-2)
    assert roofline.bound_of(roofline.Work(bytes=1e12, flops=1.0), peaks) == "hbm"
    lin = roofline.linear_work(np.array([0, 1, -1, 1]), K=64, N=32, r=16)
    assert lin.bytes == 32 * 64 * 2 + 2 * (16 * 64 + 32 * 16) * 2 + 4 * 64 * 2 + 4 * 32 * 2 + 4 * 4
    assert lin.flops == 4 * 2 * 32 * 64 + 3 * 2 * (64 * 16 + 16 * 32)
