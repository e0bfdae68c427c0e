"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code path.

* a hand-derived closed-form example (tests/golden/forward_closed_form.json)
  and a hand-worked align example (tests/golden/align_hand.json);
* a scalar brute force (pure-Python loops, math.exp) on tiny shapes;
* the merged-weight identity x(W + AB) = xW + xAB (LoRA merged into the base
  weights, as the hybrid-attention decoder page does before serving);
* adapter -1 and B = 0 both reduce the layer to the plain MoE;
* one expert, top-1, weight 1 reduces the layer to a dense two-projection MLP,
  and the dense linear to x W^T + per-adapter LoRA;
* linearity of the combine in the gate weights (one-hot weights isolate one
  expert);
* the align step against a counting sort and its invariants;
* the router against a two-expert closed form and a library top-k;
* per-token independence (any subset of tokens gives the matching rows);
* the bf16 -> float64 widening against the format's definition.

The last tests plant mistakes in the oracle (on the CPU): monkeypatched
helpers, and 21 source-level rewrites of single expressions (swapped gate/up
halves, LoRA shared across experts, a dropped gate weight, a wrong index or
comparison in the align, ...).  Each must make at least one pin fail.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import moe_lora_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _silu(v):
    return v / (1.0 + math.exp(-v))


# ----------------------------------------------------------------- fixtures
def _rand_layer(rng, T, H, I, E, k, L, r, none=True, scale=1.0):
    x = rng.standard_normal((T, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
    w = rng.random((T, k)) + 0.1
    w /= w.sum(1, keepdims=True) if T else 1
    lo = -1 if none else 0
    lora = rng.integers(lo, L, size=T) if L else np.full(T, -1)
    Wgu = rng.standard_normal((E, 2 * I, H)) * scale
    Wd = rng.standard_normal((E, H, I)) * scale
    Agu = rng.standard_normal((L, E, r, H))
    Bgu = rng.standard_normal((L, E, 2 * I, r))
    Ad = rng.standard_normal((L, E, r, I))
    Bd = rng.standard_normal((L, E, H, r))
    return dict(x=x, topk_ids=ids, topk_weights=w, lora_ids=lora, W_gate_up=Wgu,
                W_down=Wd, A_gu=Agu, B_gu=Bgu, A_d=Ad, B_d=Bd)


def _brute(d):
    """Scalar restatement: per token, per routed pair, explicit index sums."""
    x, ids, w, lora = d["x"], d["topk_ids"], d["topk_weights"], d["lora_ids"]
    Wgu, Wd = d["W_gate_up"], d["W_down"]
    T, H = x.shape
    k = ids.shape[1]
    I = Wd.shape[2]
    r = d["A_gu"].shape[2] if d["A_gu"].size else 0
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        a = int(lora[t])
        for j in range(k):
            e = int(ids[t, j])
            g = [sum(x[t, h] * Wgu[e, c, h] for h in range(H)) for c in range(2 * I)]
            if a >= 0:
                z = [sum(x[t, h] * d["A_gu"][a, e, q, h] for h in range(H)) for q in range(r)]
                for c in range(2 * I):
                    g[c] += sum(z[q] * d["B_gu"][a, e, c, q] for q in range(r))
            act = [_silu(g[i]) * g[I + i] for i in range(I)]
            dd = [sum(act[i] * Wd[e, h, i] for i in range(I)) for h in range(H)]
            if a >= 0:
                z2 = [sum(act[i] * d["A_d"][a, e, q, i] for i in range(I)) for q in range(r)]
                for h in range(H):
                    dd[h] += sum(z2[q] * d["B_d"][a, e, h, q] for q in range(r))
            for h in range(H):
                out[t][h] += w[t, j] * dd[h]
    return np.array(out)


def _fwd(d, **kw):
    return ref.moe_lora_forward_ref(d["x"], d["topk_ids"], d["topk_weights"], d["lora_ids"],
                                    d["W_gate_up"], d["W_down"], d["A_gu"], d["B_gu"],
                                    d["A_d"], d["B_d"], **kw)


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# -------------------------------------------------------------------- pins
def pin_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "forward_closed_form.json")))
    d = {k: np.array(v, dtype=np.float64) for k, v in g.items()
         if k not in ("source", "layout", "derivation")}
    d["topk_ids"] = d["topk_ids"].astype(int)
    d["lora_ids"] = d["lora_ids"].astype(int)
    out = _fwd(d)
    act0 = _silu(2.5) * 2
    act1 = _silu(4.0) * 1
    out0 = [0.75 * 2 * act0, 0.75 * 2 * act0 + 0.25 * 0.5 * act1]
    b1 = _silu(-1.0) * -0.5
    b0 = _silu(0.5) * -1.0
    out1 = [0.5 * -b1 + 0.5 * b0, 0.5 * 0.5 * b1 + 0.5 * 2 * b0]
    return np.abs(out - np.array([out0, out1])).max() < 1e-14


def pin_brute_force(seed=0):
    rng = np.random.default_rng(seed)
    ok = True
    for (T, H, I, E, k, L, r) in [(5, 6, 3, 4, 2, 3, 2), (3, 4, 5, 3, 3, 2, 1), (4, 3, 2, 2, 1, 1, 3)]:
        d = _rand_layer(rng, T, H, I, E, k, L, r)
        ok &= _rel(_fwd(d), _brute(d)) < 1e-12
    return bool(ok)


def pin_merged_identity(seed=1):
    """x(W + AB) = xW + xAB for both projections: merge each adapter into each
    expert's weights (stored layout: W' = W + B @ A) and run without LoRA."""
    rng = np.random.default_rng(seed)
    d = _rand_layer(rng, T=24, H=12, I=10, E=4, k=2, L=3, r=4)
    out = _fwd(d)
    ok = True
    for a in range(-1, 3):
        m = np.nonzero(d["lora_ids"] == a)[0]
        if not len(m):
            continue
        dm = dict(d)
        if a >= 0:
            dm["W_gate_up"] = d["W_gate_up"] + np.einsum("ecq,eqh->ech", d["B_gu"][a], d["A_gu"][a])
            dm["W_down"] = d["W_down"] + np.einsum("ehq,eqi->ehi", d["B_d"][a], d["A_d"][a])
        dm["lora_ids"] = np.full_like(d["lora_ids"], -1)
        ok &= _rel(_fwd(dm, tokens=m), out[m]) < 1e-12
    return bool(ok)


def pin_base_moe(seed=2):
    """Adapter -1 everywhere, or B = 0, gives the plain MoE (computed here by
    torch's float64 matmul per pair, a library routine)."""
    import torch
    rng = np.random.default_rng(seed)
    d = _rand_layer(rng, T=20, H=16, I=8, E=5, k=3, L=2, r=4)
    dn = dict(d, lora_ids=np.full(20, -1))
    dz = dict(d, B_gu=np.zeros_like(d["B_gu"]), B_d=np.zeros_like(d["B_d"]))
    x = torch.tensor(d["x"])
    exp = torch.zeros(20, 16, dtype=torch.float64)
    for t in range(20):
        for j in range(3):
            e = int(d["topk_ids"][t, j])
            g = torch.tensor(d["W_gate_up"][e]) @ x[t]
            act = torch.nn.functional.silu(g[:8]) * g[8:]
            exp[t] += float(d["topk_weights"][t, j]) * (torch.tensor(d["W_down"][e]) @ act)
    exp = exp.numpy()
    return bool(_rel(_fwd(dn), exp) < 1e-12 and _rel(_fwd(dz), exp) < 1e-12)


def pin_dense_reduction(seed=3):
    """E = 1, top-1, weight 1: the layer is a dense two-projection MLP with
    per-token LoRA; the dense linear is x W^T + (x A^T) B^T per adapter."""
    rng = np.random.default_rng(seed)
    d = _rand_layer(rng, T=9, H=6, I=5, E=1, k=1, L=3, r=2)
    d["topk_weights"] = np.ones((9, 1))
    y_gu = ref.moe_lora_linear_ref(d["x"], d["lora_ids"], d["W_gate_up"][0],
                                   d["A_gu"][:, 0], d["B_gu"][:, 0])
    act = np.array([[_silu(v) for v in row[:5]] for row in y_gu]) * y_gu[:, 5:]
    y_d = ref.moe_lora_linear_ref(act, d["lora_ids"], d["W_down"][0], d["A_d"][:, 0], d["B_d"][:, 0])
    ok = _rel(_fwd(d), y_d) < 1e-12
    # dense linear against explicit per-token sums
    x, W, A, B, lo = d["x"], d["W_gate_up"][0], d["A_gu"][:, 0], d["B_gu"][:, 0], d["lora_ids"]
    exp = np.zeros((9, 10))
    for t in range(9):
        for n in range(10):
            s = sum(x[t, h] * W[n, h] for h in range(6))
            if lo[t] >= 0:
                s += sum(sum(x[t, h] * A[lo[t], q, h] for h in range(6)) * B[lo[t], n, q]
                         for q in range(2))
            exp[t, n] = s
    ok &= _rel(y_gu, exp) < 1e-12
    return bool(ok)


def pin_linearity(seed=4):
    rng = np.random.default_rng(seed)
    d = _rand_layer(rng, T=10, H=8, I=6, E=4, k=2, L=2, r=2)
    out = _fwd(d)
    ok = _rel(_fwd(dict(d, topk_weights=3.0 * d["topk_weights"])), 3.0 * out) < 1e-13
    # one-hot: only j=0 counts -> equals the top-1 layer on the first expert
    oh = np.zeros_like(d["topk_weights"])
    oh[:, 0] = 1.0
    d1 = dict(d, topk_ids=d["topk_ids"][:, :1], topk_weights=np.ones((10, 1)))
    ok &= _rel(_fwd(dict(d, topk_weights=oh)), _fwd(d1)) < 1e-13
    return bool(ok)


def _counting_sort_align(topk_ids, lora_ids, E, L, bm):
    """Align restated as a stable counting sort: walk entries in flat order,
    append each to its (expert, adapter) bucket, then lay the buckets out."""
    T, k = topk_ids.shape
    buckets = {(e, a): [] for e in range(E) for a in range(-1, L)}
    for f in range(T * k):
        buckets[(int(topk_ids[f // k, f % k]), int(lora_ids[f // k]))].append(f)
    sorted_ids, blk, seg = [], [], []
    for e in range(E):
        run = []
        for a in range(-1, L):
            seg.append(len(sorted_ids) + len(run))
            run += buckets[(e, a)]
        padded = run + [T * k] * ((-len(run)) % bm)
        sorted_ids += padded
        blk += [e] * (len(padded) // bm)
    seg.append(len(sorted_ids))
    return sorted_ids, blk, seg


def pin_align(seed=5):
    g = json.load(open(os.path.join(GOLDEN, "align_hand.json")))
    ok = True
    for c in g["cases"]:
        out = ref.align_ref(np.array(c["topk_ids"]), np.array(c["lora_ids"]), c["E"], c["L"], c["block_m"])
        ok &= out["sorted_ids"].tolist() == c["sorted_ids"]
        ok &= out["blk_expert"].tolist() == c["blk_expert"]
        ok &= out["seg_off"].tolist() == c["seg_off"]
        ok &= out["num_post_pad"] == c["num_post_pad"]
    rng = np.random.default_rng(seed)
    for (T, k, E, L, bm) in [(50, 2, 8, 4, 16), (33, 3, 5, 2, 4), (1, 1, 1, 1, 8), (64, 4, 16, 3, 1)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        lo = rng.integers(-1, L, size=T)
        out = ref.align_ref(ids, lo, E, L, bm)
        s, b, sg = _counting_sort_align(ids, lo, E, L, bm)
        ok &= out["sorted_ids"].tolist() == s and out["blk_expert"].tolist() == b
        ok &= out["seg_off"].tolist() == sg
        # invariants
        si = out["sorted_ids"]
        ok &= sorted(si[si < T * k].tolist()) == list(range(T * k))
        ok &= out["num_post_pad"] % bm == 0
        ok &= bool(np.all(np.diff(out["blk_expert"]) >= 0))
    return bool(ok)


def pin_router(seed=6):
    """Router: closed form for two experts (weights are a logistic of the logit
    gap), a library top-k (torch.topk over softmax in float64) on continuous
    logits, ties broken by the lower index, and the invariants."""
    import torch
    ok = True
    ids, w = ref.router_topk_ref(np.array([[0.5, 2.0]], dtype=np.float32), 2)
    ok &= ids.tolist() == [[1, 0]]
    ok &= abs(w[0, 0] - 1.0 / (1.0 + math.exp(-1.5))) < 1e-15
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((40, 16)).astype(np.float32)
    ids, w = ref.router_topk_ref(lg, 4)
    p = torch.softmax(torch.tensor(lg, dtype=torch.float64), -1)
    tv, ti = torch.topk(p, 4, -1)
    ok &= np.array_equal(ids, ti.numpy())
    ok &= np.abs(w - (tv / tv.sum(-1, keepdim=True)).numpy()).max() < 1e-14
    ok &= np.allclose(w.sum(1), 1.0) and bool(np.all(np.diff(w, axis=1) <= 0))
    tie = np.array([[1.0, 3.0, 3.0, 1.0, 3.0]], dtype=np.float32)
    ok &= ref.router_topk_ref(tie, 3)[0].tolist() == [[1, 2, 4]]
    ok &= ref.router_topk_ref(tie, 4)[0].tolist() == [[1, 2, 4, 0]]
    return bool(ok)


def pin_token_subset(seed=7):
    """Each token's output depends only on its own routing and adapter: any
    subset of tokens, in any order, gives the matching rows of the full
    evaluation (with adapters, so a per-token index slip shows)."""
    rng = np.random.default_rng(seed)
    d = _rand_layer(rng, T=12, H=8, I=6, E=4, k=2, L=2, r=2)
    full = _fwd(d)
    ok = True
    for sub in ([7, 2, 11], [11, 10, 9, 8], [0]):
        ok &= _rel(_fwd(d, tokens=sub), full[sub]) < 1e-13
    return bool(ok)


def pin_bf16_conversion():
    """bf16 bit patterns widen exactly: the value is the float32 whose upper
    16 bits are the pattern (sign, 8-bit exponent, 7-bit mantissa)."""
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001], dtype=np.uint16)
    exp = [1.0, -1.0, 3.140625, 0.0, -0.0, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133]
    got = ref.as_f64(bits).tolist()
    return got == exp and math.copysign(1.0, got[4]) == -1.0


PINS = [pin_closed_form, pin_brute_force, pin_merged_identity, pin_base_moe,
        pin_dense_reduction, pin_linearity, pin_align, pin_router, pin_token_subset,
        pin_bf16_conversion]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    assert pin()


def test_oracle_rejects_bad_ids():
    rng = np.random.default_rng(8)
    d = _rand_layer(rng, T=4, H=4, I=2, E=3, k=1, L=2, r=1)
    with pytest.raises(ValueError):
        _fwd(dict(d, topk_ids=np.full((4, 1), 3)))
    with pytest.raises(ValueError):
        _fwd(dict(d, lora_ids=np.array([0, 1, 2, -1])))
    with pytest.raises(ValueError):
        ref.align_ref(np.array([[0], [5]]), np.array([0, 0]), 3, 2, 4)


# ------------------------------------------------------ planted mistakes
def _mut_silu_sign(v):
    return v / (1.0 + np.exp(v))


def _mut_drop_lora(X, A, B):
    return np.zeros((X.shape[0], B.shape[0]))


def _mut_lora_transpose(X, A, B):
    z = X @ A.T
    return (z @ B.T) * 0.5 + (z @ B.T)[:, ::-1] * 0.5


MUTATIONS = [("silu", _mut_silu_sign), ("_lora_delta", _mut_drop_lora),
             ("_lora_delta", _mut_lora_transpose)]


@pytest.mark.parametrize("name,mut", MUTATIONS, ids=["silu_sign", "drop_lora", "scramble_lora"])
def test_pins_catch_planted_mistakes(monkeypatch, name, mut):
    monkeypatch.setattr(ref, name, mut)
    results = {p.__name__: p() for p in PINS if p is not pin_align}
    assert not all(results.values()), results


def test_pins_catch_align_mistake(monkeypatch):
    orig = np.lexsort
    # drop the flat-index tie break (unstable order within a segment)
    monkeypatch.setattr(np, "lexsort", lambda keys: orig((-keys[0],) + tuple(keys[1:])))
    assert not pin_align()


# ------------------------------------------------ source-level mutations
# Each mutation rewrites one expression of the oracle's source (a swapped
# operand, a dropped term, a wrong index or comparison) and runs every pin on
# the rewritten module: at least one pin must fail or raise.
ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "moe_lora_ref.py")

SOURCE_MUTATIONS = {
    "gate_up_halves_swapped": ("act = silu(g[:, :I]) * g[:, I:]", "act = silu(g[:, I:]) * g[:, :I]"),
    "silu_on_both_halves": ("act = silu(g[:, :I]) * g[:, I:]", "act = silu(g[:, :I]) * silu(g[:, I:])"),
    "gu_lora_shared_across_experts": ("as_f64(A_gu[a, e]), as_f64(B_gu[a, e])",
                                      "as_f64(A_gu[a, 0]), as_f64(B_gu[a, 0])"),
    "d_lora_shared_across_experts": ("as_f64(A_d[a, e]), as_f64(B_d[a, e])",
                                     "as_f64(A_d[a, 0]), as_f64(B_d[a, 0])"),
    "down_lora_reads_gate": ("_lora_delta(act[m],", "_lora_delta(g[m][:, :I],"),
    "down_lora_dropped": ("d[m] += _lora_delta(act[m]", "d[m] += 0 * _lora_delta(act[m]"),
    "gate_up_lora_after_activation": ("g[m] += _lora_delta(Xe[m]", "g[m] += 0 * _lora_delta(Xe[m]"),
    "gate_weight_dropped": ("out[i] += topk_weights[t, j] * pair_d[(i, j)]", "out[i] += pair_d[(i, j)]"),
    "gate_weight_of_first_expert": ("out[i] += topk_weights[t, j] *", "out[i] += topk_weights[t, 0] *"),
    "adapter_indexed_by_subset_row": ("ae = lora_ids[tokens[rows]]", "ae = lora_ids[rows]"),
    "token_indexed_by_subset_row": ("Xe = x[tokens[rows]]", "Xe = x[rows]"),
    "expand_uses_shrink_matrix": ("return z @ B.T", "return z @ A[:, :B.shape[0]].T if A.shape[1] >= B.shape[0] else z @ B.T"),
    "bf16_bits_misplaced": ("<< 16", "<< 15"),
    "silu_sign": ("v / (1.0 + np.exp(-v))", "v / (1.0 + np.exp(v))"),
    "align_unstable": ("np.lexsort((f_of, a_of + 1, e_of))", "np.lexsort((-f_of, a_of + 1, e_of))"),
    "align_adapters_reversed": ("np.lexsort((f_of, a_of + 1, e_of))", "np.lexsort((f_of, -a_of, e_of))"),
    "align_seg_off_inclusive": ("np.count_nonzero(a_of[mine] < a)", "np.count_nonzero(a_of[mine] <= a)"),
    "align_exact_multiple_overpadded": ("pad = -(-count // block_m) * block_m",
                                        "pad = (count // block_m + 1) * block_m"),
    "router_ties_to_higher_index": ("(-float(logits[t, e]), e)", "(-float(logits[t, e]), -e)"),
    "router_weights_not_renormalised": ("w[t] = sel / sel.sum()", "w[t] = sel / np.exp(lt - lt.max()).sum()"),
    "linear_adapter_ignored": ("_lora_delta(x[m], as_f64(A[a]), as_f64(B[a]))",
                               "_lora_delta(x[m], as_f64(A[0]), as_f64(B[0]))"),
}


def _oracle_from_source(src):
    import types
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, ORACLE_SRC, "exec"), mod.__dict__)
    return mod


def _run_pins(monkeypatch, mod):
    import sys
    monkeypatch.setattr(sys.modules[__name__], "ref", mod)
    results = {}
    for p in PINS:
        try:
            results[p.__name__] = bool(p())
        except Exception as exc:            # a mutant that raises is caught too
            results[p.__name__] = f"raised {type(exc).__name__}"
    return results


def test_unmutated_source_passes_every_pin(monkeypatch):
    res = _run_pins(monkeypatch, _oracle_from_source(open(ORACLE_SRC).read()))
    assert all(v is True for v in res.values()), res


@pytest.mark.parametrize("name", sorted(SOURCE_MUTATIONS))
def test_pins_catch_source_mutation(monkeypatch, name):
    old, new = SOURCE_MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    res = _run_pins(monkeypatch, _oracle_from_source(src.replace(old, new)))
    assert not all(v is True for v in res.values()), res


# ------------------------------------------------ property test (hypothesis)
def test_oracle_matches_brute_force_on_random_tiny_layers():
    """The oracle against the scalar brute force on layers drawn by
    hypothesis: sizes, routing (duplicates allowed), adapters including -1,
    LoRA on or off."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=40, deadline=None, derandomize=True)
    @hyp.given(st.integers(0, 5), st.integers(1, 6), st.integers(1, 5), st.integers(1, 4),
               st.integers(1, 3), st.integers(0, 3), st.integers(1, 3), st.integers(0, 2 ** 31 - 1))
    def check(T, H, I, E, k, L, r, seed):
        rng = np.random.default_rng(seed)
        d = _rand_layer(rng, T, H, I, E, min(k, E), L, r)
        if T:
            d["topk_ids"] = rng.integers(0, E, size=(T, min(k, E)))   # duplicates allowed
        got = _fwd(d)
        exp = _brute(d)
        assert got.shape == (T, H)
        if T:
            assert _rel(got, exp) < 1e-12

    check()
