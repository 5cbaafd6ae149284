"""Pins for oracle.route: brute force, library top-k/softmax, structural invariants."""

import numpy as np
import torch

import synth
from oracle import route


def _brute_topk(row, k):
    return [e for _, e in sorted((-float(v), e) for e, v in enumerate(row))[:k]]


def test_topk_brute_force_with_forced_ties():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((64, 16)).astype(np.float32)
    # plant ties, including the k-th boundary and equal maxima
    logits[::3, 5] = logits[::3, 2]
    logits[1::4, :] = np.round(logits[1::4, :])
    logits[2, :] = 0.5
    logits[4, 7] = -0.0
    logits[4, 3] = 0.0
    for k in (1, 2, 4, 8):
        ids = route.topk_ids(logits, k)
        for t in range(64):
            assert ids[t].tolist() == _brute_topk(logits[t], k)
    assert route.topk_ids(logits, 4)[2].tolist() == [0, 1, 2, 3]


def test_topk_matches_torch_on_tie_free_data():
    l = synth.gen_logits(512, 256)
    ids = route.topk_ids(l.numpy(), 8)
    ref = torch.topk(l, 8, dim=1, sorted=True).indices.numpy()
    assert np.array_equal(ids, ref)


def test_gates_renormalised_softmax():
    l = synth.gen_logits(300, 256).numpy()
    ids, g, _, _ = route.plan(l, 8)
    assert np.max(np.abs(g.sum(axis=1) - 1.0)) < 1e-12
    assert np.all(np.diff(g, axis=1) <= 0)          # descending logits -> descending gates
    # library: softmax over all experts, take the chosen ones, renormalise
    sm = torch.softmax(torch.from_numpy(l).double(), dim=1).numpy()
    chosen = np.take_along_axis(sm, ids.astype(np.int64), axis=1)
    assert np.max(np.abs(chosen / chosen.sum(axis=1, keepdims=True) - g)) < 1e-12
    _, g1, _, _ = route.plan(l, 1)
    assert np.all(g1 == 1.0)


def test_permutation_and_offsets_invariants():
    rng = np.random.default_rng(8)
    for T, E, k in [(4, 8, 2), (1, 256, 8), (100, 16, 4), (0, 8, 2)]:
        l = rng.standard_normal((T, E)).astype(np.float32)
        ids, _, perm, off = route.plan(l, k)
        S = T * k
        assert off.shape == (E + 1,) and off[0] == 0 and off[E] == S
        assert sorted(perm.tolist()) == list(range(S))                # bijection
        flat = ids.reshape(-1)
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert np.all(flat[seg] == e)                             # grouped by expert
            assert np.all(np.diff(seg) > 0)                           # stable: ascending slot
        assert np.array_equal(np.diff(off), np.bincount(flat, minlength=E))


def test_tiny_route_fixture():
    # row 2 lists a higher id first: its larger logit is at expert 3
    l = np.array([[0.1, 0.9, 0.3, 0.9], [2.0, -1.0, 0.0, 1.0], [0.0, 0.5, -1.0, 3.0]], dtype=np.float32)
    ids, g, perm, off = route.plan(l, 2)
    assert ids.tolist() == [[1, 3], [0, 3], [3, 1]]
    assert np.allclose(g[0], [0.5, 0.5], atol=0, rtol=0)
    e = np.exp(-1.0)
    assert np.allclose(g[1], [1 / (1 + e), e / (1 + e)], rtol=1e-15)
    e = np.exp(-2.5)
    assert np.allclose(g[2], [1 / (1 + e), e / (1 + e)], rtol=1e-15)
    # slots: 0->e1, 1->e3, 2->e0, 3->e3, 4->e3, 5->e1
    assert perm.tolist() == [2, 0, 5, 1, 3, 4]
    assert off.tolist() == [0, 1, 3, 3, 6]
