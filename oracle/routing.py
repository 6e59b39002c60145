"""Init-routing (oracle).  Test infrastructure only.

Sources:
* Qwen3-MoE low-latency inference practice, section "GMM enablement and
  routing optimisation": init-routing produces the expert sort order of the
  token-expert pairs; compute-expert-tokens gives the number of tokens each
  expert must process.
* Hy3 295B MoE practice, section 6.2: the grouped matmul's ``group_list`` is
  the per-expert token count.

Notation: pair p = t*k + j (token t, top-k slot j); pos = index in expert-sorted
order.  Reading (the pages do not fix it): inside one expert's segment pairs
keep ascending p (a stable sort).
"""
from __future__ import annotations

import numpy as np


def init_routing(topk_idx, E: int):
    """Returns counts[E], offsets[E+1], sorted_pair[P] (pos -> p), pair_pos[P] (p -> pos), all int32."""
    idx = np.asarray(topk_idx, np.int64).reshape(-1)
    P = idx.size
    if P and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.bincount(idx, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, np.int32)
    np.cumsum(counts, out=offsets[1:])
    sorted_pair = np.argsort(idx, kind="stable").astype(np.int32)
    pair_pos = np.empty(P, np.int32)
    pair_pos[sorted_pair] = np.arange(P, dtype=np.int32)
    return counts, offsets, sorted_pair, pair_pos


def expand_rows(x, sorted_pair, k: int):
    """x_exp[pos] = x[sorted_pair[pos] // k]: the token rows in expert-sorted order."""
    return np.asarray(x)[np.asarray(sorted_pair, np.int64) // k]


def init_routing_range(topk_idx, E: int, e0: int, e1: int):
    """Init-routing restricted to the local experts [e0, e1) (Qwen3-MoE practice, MoE EP with
    AllGather + ReduceScatter: init_routing_v2 keeps only the tokens of the experts in this rank's
    range).  Local expert l = e - e0.

    Returns counts[e1-e0], offsets[e1-e0+1], sorted_pair[P_loc] (the local pairs, by local expert,
    ascending p inside one), pair_pos[P] (p -> pos, -1 for a pair whose expert is not local).
    """
    if not 0 <= e0 < e1 <= E:
        raise ValueError("need 0 <= e0 < e1 <= E")
    idx = np.asarray(topk_idx, np.int64).reshape(-1)
    P = idx.size
    if P and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    local = (idx >= e0) & (idx < e1)
    p_loc = np.nonzero(local)[0]                       # ascending pair index
    lidx = idx[p_loc] - e0
    counts = np.bincount(lidx, minlength=e1 - e0).astype(np.int32)
    offsets = np.zeros(e1 - e0 + 1, np.int32)
    np.cumsum(counts, out=offsets[1:])
    sorted_pair = p_loc[np.argsort(lidx, kind="stable")].astype(np.int32)
    pair_pos = np.full(P, -1, np.int32)
    pair_pos[sorted_pair] = np.arange(sorted_pair.size, dtype=np.int32)
    return counts, offsets, sorted_pair, pair_pos
