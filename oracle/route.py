"""Routing oracle: top-k ids, renormalised gates, token permutation, expert offsets.

TEST INFRASTRUCTURE ONLY: see the package docstring.

[P1] "How it works" says both tiers run off one shared route geometry and
accumulate into one topk_sum. [P2] "Summary" says the same. Neither page
defines the routing function. This module takes the plainest reading,
softmax top-k with the chosen gates renormalised:

1. For each token t, the k experts with the largest router logit, in order
   of descending logit. Equal logits go to the lower expert id. Softmax is
   monotonic, so this is the same set as top-k of the softmax. Selecting on
   the raw logits keeps the choice free of exp rounding.
2. gates[t, j] = exp(l_j - l_max) / sum over the chosen experts of
   exp(l_i - l_max). This equals softmax followed by renormalisation over the
   k chosen experts.
3. perm is the stable sort of the flat slot indices s = t*k + j by expert id.
   Within one expert the slots keep ascending s.
4. offsets[e] is the exclusive prefix sum of the per-expert slot counts.
   offsets[E] = T*k.
"""

import numpy as np


def topk_ids(logits, k):
    """int32 [T, k]: the k largest logits per row, descending, ties to the lower id."""
    l = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gates(logits, ids):
    """float64 [T, k]: softmax over the chosen logits (the renormalised gates)."""
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    chosen = np.take_along_axis(l, np.asarray(ids, dtype=np.int64), axis=1)
    z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def permutation(ids, E):
    """(perm int32 [T*k], offsets int32 [E+1]): stable counting sort of slots by expert."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return perm, offsets


def plan(logits, k):
    """All route outputs at once: ids, gates, perm, offsets."""
    l = np.asarray(logits, dtype=np.float32)
    E = l.shape[1]
    ids = topk_ids(l, k)
    g = gates(l, ids)
    perm, offsets = permutation(ids, E)
    return ids, g, perm, offsets
