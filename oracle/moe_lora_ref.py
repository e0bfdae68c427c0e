"""CPU oracle for the fused MoE-LoRA expert layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference arm of ``bench.py`` may import this module.  The library's product
path never calls it, and it shares no code with the CUDA path.

It is a plain, slow, obviously correct statement of what the layer computes,
in float64 (every bf16 input converts to float64 exactly).  The passages it
follows are on the multi-LoRA MoE serving blog (vllm.com.cn/blog/multi-lora):

* "Implementing multi-LoRA for MoE in vLLM" (the expert FFN paragraph): each
  expert is a small fully connected network; its gate_up projection expands
  the hidden state to the intermediate space and its down projection maps
  it back; vLLM's fused_moe runs one GEMM per expert over the tokens routed
  to it.  A LoRA adapter keeps W frozen and adds x A B with A of shape
  h_in x r and B of shape r x h_out, so y = xW + xAB; the shrink is z = xA
  and the expand multiplies z by B.
* Same section, the paragraph after Fig. 1: every expert gets its own four
  LoRA operations (gate_up shrink/expand, down shrink/expand), per expert and
  per adapter; the router sends each token to its experts and the experts'
  outputs are aggregated (weighted by the router's top-k gate weights).
* The layer's activation between the projections is SiLU(gate) * up, with the
  first I rows of the gate_up weight giving `gate` and the last I rows `up`.

Readings taken where the pages are silent (each also listed in the design
notes): LoRA scale 1, no bias, adapter id -1 = no LoRA on either projection,
one LoRA pair for the fused gate_up weight, topk weights used as given.

Storage convention: the weights are stored "out x in" (row-major, the
reduction axis contiguous), so the page's W (h_in x h_out) is the transpose
of the stored matrix: y = x @ W_stored.T.  The same holds for A (stored r x
h_in) and B (stored h_out x r).

Pins (tests under ``tests/test_oracle_pins.py``): a hand-derived closed-form
example, a scalar brute force on tiny shapes, the merged-weight identity
x(W + AB) = xW + xAB, adapter -1 / B = 0 reducing to the plain MoE, E = 1
top-1 reducing to a dense two-projection MLP, linearity in the gate weights,
the align definition checked by a counting sort and its invariants, the
router against a two-expert closed form and a library top-k, per-token
independence, and the bf16 widening against the format's definition.  The
same tests rewrite single expressions of this file (swapped operands, dropped
terms, wrong indices) and check that some pin fails for each rewrite.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64", "align_ref", "moe_lora_forward_ref", "moe_lora_linear_ref",
    "router_topk_ref", "silu",
]


def as_f64(a):
    """bf16 bit patterns (uint16/int16) or any float array -> float64 (exact)."""
    a = np.asarray(a)
    if a.dtype in (np.uint16, np.int16):
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def silu(v):
    """SiLU(v) = v * sigmoid(v) = v / (1 + exp(-v))."""
    return v / (1.0 + np.exp(-v))


def align_ref(topk_ids, lora_ids, E, L, block_m):
    """The align step: group the T*k routed entries by (expert, adapter).

    Definition (multi-LoRA MoE blog, "Implementing multi-LoRA for MoE": the
    fused_moe_lora kernel follows fused_moe's per-expert grouping and adds one
    grid dimension over the active adapters):

    * entry f = t*k + j has expert e = topk_ids[t, j] and adapter
      a = lora_ids[t];
    * entries are ordered by the key (e, a + 1, f) -- adapter -1 first, ties
      broken by the flat index, so the order is stable;
    * each expert's run of entries is padded with the sentinel T*k up to a
      multiple of ``block_m``; an expert with no entries gets no block;
    * blk_expert[b] is the expert owning block b; seg_off[e*(L+1) + a+1] is the
      position of the first entry of segment (e, a) and seg_off[-1] = P, the
      padded total (num_post_pad).
    """
    topk_ids = np.asarray(topk_ids, dtype=np.int64)
    lora_ids = np.asarray(lora_ids, dtype=np.int64)
    T, k = topk_ids.shape
    n = T * k
    e_of = topk_ids.reshape(-1)
    a_of = np.repeat(lora_ids, k)
    f_of = np.arange(n)
    if n and (e_of.min() < 0 or e_of.max() >= E):
        raise ValueError("expert id out of range")
    if n and (a_of.min() < -1 or a_of.max() >= L):
        raise ValueError("adapter id out of range")

    order = np.lexsort((f_of, a_of + 1, e_of))          # last key is primary
    count = np.bincount(e_of, minlength=E)
    pad = -(-count // block_m) * block_m
    start = np.concatenate([[0], np.cumsum(pad)])
    P = int(start[-1])

    sorted_ids = np.full(P, n, dtype=np.int64)
    blk_expert = np.zeros(P // block_m, dtype=np.int64)
    seg_off = np.zeros(E * (L + 1) + 1, dtype=np.int64)
    pos = 0
    for e in range(E):
        mine = order[pos:pos + count[e]]
        sorted_ids[start[e]:start[e] + count[e]] = mine
        blk_expert[start[e] // block_m:start[e + 1] // block_m] = e
        for a in range(-1, L):
            seg_off[e * (L + 1) + a + 1] = start[e] + np.count_nonzero(a_of[mine] < a)
        pos += count[e]
    seg_off[-1] = P
    return {"sorted_ids": sorted_ids, "blk_expert": blk_expert, "seg_off": seg_off,
            "num_post_pad": P}


def router_topk_ref(logits, k):
    """The router step upstream of the layer (multi-LoRA MoE blog, "Implementing
    multi-LoRA for MoE in vLLM": the routing algorithm sends each token to its
    most relevant experts, whose outputs are then aggregated).

    Plain definition: p = softmax(logits[t]); the k experts with the largest p
    are chosen, larger first, the lower expert index first among equal values;
    their gate weights are p renormalised over the chosen k, i.e. the softmax
    of the chosen logits.  Softmax is monotonic, so the choice is taken on the
    logits themselves (the same values and precision the GPU compares).
    Returns (ids [T,k] int64, weights [T,k] float64)."""
    logits = np.asarray(logits)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("k out of range")
    ids = np.zeros((T, k), dtype=np.int64)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        ids[t] = order
        lt = logits[t].astype(np.float64)
        sel = np.exp(lt[order] - lt.max())
        w[t] = sel / sel.sum()
    return ids, w


def _lora_delta(X, A, B):
    """The two LoRA steps of the blog's y = xW + xAB: shrink z = xA, expand zB
    (A stored r x h_in, B stored h_out x r)."""
    z = X @ A.T
    return z @ B.T


def moe_lora_forward_ref(x, topk_ids, topk_weights, lora_ids, W_gate_up, W_down,
                         A_gu=None, B_gu=None, A_d=None, B_d=None, tokens=None,
                         return_pairs=False):
    """out[t] = sum_j topk_weights[t,j] * expert_{e_tj, a_t}(x[t]), float64.

    For one routed pair (token t, expert e, adapter a):
      g   = x W_gu[e]^T + [a >= 0] (x A_gu[a,e]^T) B_gu[a,e]^T      (2I values)
      act = SiLU(g[:I]) * g[I:]
      d   = act W_d[e]^T + [a >= 0] (act A_d[a,e]^T) B_d[a,e]^T     (H values)
    and the token's output is the gate-weighted sum of its k pairs, j
    ascending.  Each expert is evaluated as one GEMM over its tokens (the
    fused_moe grouping), each adapter's LoRA over that adapter's tokens.

    ``tokens``: optional subset of token indices to evaluate (the output rows
    follow that order); each token's output depends only on its own routing.
    """
    x = as_f64(x)
    topk_ids = np.asarray(topk_ids, dtype=np.int64)
    topk_weights = np.asarray(topk_weights, dtype=np.float64)
    lora_ids = np.asarray(lora_ids, dtype=np.int64)
    T, k = topk_ids.shape
    E = W_gate_up.shape[0]
    H = x.shape[1]
    I = W_down.shape[2]
    L = 0 if A_gu is None else A_gu.shape[0]
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, dtype=np.int64)
    if topk_ids.size and (topk_ids.min() < 0 or topk_ids.max() >= E):
        raise ValueError("expert id out of range")
    if lora_ids.size and (lora_ids.min() < -1 or lora_ids.max() >= L):
        raise ValueError("adapter id out of range")

    pair_d = {}                       # (row in `tokens`, j) -> d (H values)
    pair_act = {}
    sub_ids = topk_ids[tokens]
    for e in np.unique(sub_ids):
        rows, js = np.nonzero(sub_ids == e)
        Xe = x[tokens[rows]]
        Wgu = as_f64(W_gate_up[e])
        Wd = as_f64(W_down[e])
        g = Xe @ Wgu.T
        ae = lora_ids[tokens[rows]]
        for a in np.unique(ae[ae >= 0]):
            m = ae == a
            g[m] += _lora_delta(Xe[m], as_f64(A_gu[a, e]), as_f64(B_gu[a, e]))
        act = silu(g[:, :I]) * g[:, I:]
        d = act @ Wd.T
        for a in np.unique(ae[ae >= 0]):
            m = ae == a
            d[m] += _lora_delta(act[m], as_f64(A_d[a, e]), as_f64(B_d[a, e]))
        for i in range(len(rows)):
            pair_d[(rows[i], js[i])] = d[i]
            pair_act[(rows[i], js[i])] = act[i]

    out = np.zeros((len(tokens), H), dtype=np.float64)
    for i, t in enumerate(tokens):
        for j in range(k):
            out[i] += topk_weights[t, j] * pair_d[(i, j)]
    if return_pairs:
        return out, pair_act, pair_d
    return out


def moe_lora_linear_ref(x, lora_ids, W, A=None, B=None):
    """Dense multi-LoRA linear: y[t] = x[t] W^T + [a_t >= 0] (x[t] A[a_t]^T) B[a_t]^T.

    The blog's y = xW + xAB for one projection, one adapter per token (the
    degenerate MoE layer with one expert, top-1, weight 1, no activation).
    W stored N x K, A stored [L][r][K], B stored [L][N][r]."""
    x = as_f64(x)
    lora_ids = np.asarray(lora_ids, dtype=np.int64)
    W = as_f64(W)
    y = x @ W.T
    L = 0 if A is None else A.shape[0]
    if lora_ids.size and (lora_ids.min() < -1 or lora_ids.max() >= L):
        raise ValueError("adapter id out of range")
    for a in np.unique(lora_ids[lora_ids >= 0]):
        m = lora_ids == a
        y[m] += _lora_delta(x[m], as_f64(A[a]), as_f64(B[a]))
    return y
