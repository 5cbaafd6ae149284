"""The process-pool form of the layer oracle (tests/oracle_pool.py) equals oracle.layer.moe_forward.

The pool runs the oracle's own per-expert steps in spawned workers and sums
the slots in the parent; the result must match moe_forward exactly, since
both add the same float64 terms in the same slot order.
"""

import numpy as np

import synth
from oracle import layer, route
from tests import oracle_pool

H, I, E, K = 256, 128, 8, 2


def test_pool_matches_moe_forward_exactly():
    L = synth.tiny_layer()
    T = 12
    x = synth.gen_x(T, H, seed=3).float().numpy().astype(np.float64)
    logits = synth.gen_logits(T, E, seed=3).numpy()
    ids, g, _, _ = route.plan(logits, K)
    tokens = [0, 5, 11]
    ref = layer.moe_forward(x, ids, g, L.expert_numpy, H, I, tokens=tokens)
    got = oracle_pool.moe_rows(x, ids, g, L.expert_numpy, H, I, tokens=tokens, workers=2)
    assert np.array_equal(got, ref)
    serial = oracle_pool.moe_rows(x, ids, g, L.expert_numpy, H, I, workers=1)
    assert np.array_equal(serial, layer.moe_forward(x, ids, g, L.expert_numpy, H, I))
