"""The layer oracle over many experts, spread across host processes (test infrastructure).

``oracle.layer.moe_forward`` dequantises each routed expert once, in one
process. At the 256-expert shape (H=6144, I=2048) that is about two seconds
per expert, so a parity test that reaches every expert of the layer runs the
oracle's own per-expert steps in a pool of processes instead:

1. each worker takes one expert, dequantises it with
   ``oracle.layer.expert_weights`` and applies ``oracle.layer.expert_ffn`` to
   the activation rows routed to it;
2. the parent places each result at its (token, slot) position and forms
   every token's gate-weighted sum over its k slots in slot order, as
   ``moe_forward`` does.

``tests/test_oracle_pool.py`` checks on CPU that this equals ``moe_forward``.

The pool uses the spawn start method, so a worker never inherits a CUDA
context, and each worker's BLAS runs single-threaded so that the workers do
not oversubscribe the host cores. This module imports only NumPy and the
oracle.
"""

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

from oracle import layer as olayer

_BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _expert_rows(job):
    ex, H, I, xs = job
    w13, w2 = olayer.expert_weights(ex, H, I)
    return olayer.expert_ffn(w13, w2, xs, I, act_quant=ex.get("act_quant"), act=ex.get("act", "bf16"))


def host_workers(n_jobs, cap=16):
    return max(1, min(n_jobs, cap, len(os.sched_getaffinity(0))))


def moe_rows(x, ids, gates, get_expert, H, I, tokens=None, workers=None):
    """The oracle layer output for the given tokens, float64 [len(tokens), H].

    Same definition and arguments as ``oracle.layer.moe_forward`` (all
    columns). ``get_expert(e)`` returns the expert dict in the oracle's
    numpy form; it is called in the parent, and the dict is sent to a worker.
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(ids)
    gates = np.asarray(gates, dtype=np.float64)
    T, k = ids.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    sub = ids[tokens]
    experts = [int(e) for e in np.unique(sub)]
    where = {e: np.nonzero(sub == e) for e in experts}
    jobs = [(get_expert(e), H, I, x[tokens[where[e][0]]]) for e in experts]
    n = host_workers(len(jobs)) if workers is None else workers
    if n <= 1:
        results = [_expert_rows(j) for j in jobs]
    else:
        saved = {v: os.environ.get(v) for v in _BLAS_ENV}
        for v in _BLAS_ENV:
            os.environ[v] = "1"
        try:
            with ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")) as ex:
                results = list(ex.map(_expert_rows, jobs))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old
    y = np.zeros((len(tokens), k, H), dtype=np.float64)
    for e, r in zip(experts, results):
        tl, jj = where[e]
        y[tl, jj] = r
    out = np.zeros((len(tokens), H), dtype=np.float64)
    for j in range(k):
        out += gates[tokens, j][:, None] * y[:, j]
    return out
