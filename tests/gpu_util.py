"""Helpers for the GPU tests: move a synthetic layer to the device, run the library, compare with the oracle."""

import numpy as np
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import layer as olayer
from tests import oracle_pool

# Per token row: max |out - ref| <= REL_TOL * max |ref|, with fp32 accumulation.
REL_TOL = 2e-2


def device_experts(L):
    """Expert tuples for hmoe_pack_weights. The tensors must already be on the GPU."""
    out = []
    for ex in L.experts:
        c13, s13, g13 = ex["w13"]
        c2, s2, g2 = ex["w2"]
        out.append((c13, s13, g13, c2, s2, g2))
    return out


def act_dtype(L):
    """The library's activation-type code for a synthetic layer."""
    return hm.ACT_F16 if getattr(L, "act", "bf16") == "f16" else hm.ACT_BF16


def build(L, max_tokens):
    bm = None if L.bit_map is None else [int(b) for b in L.bit_map]
    return hm.HybridMoELayer(L.H, L.I, L.E, L.topk, bm, device_experts(L), kept_format=L.kept_format,
                             max_tokens=max_tokens, act_dtype=act_dtype(L))


def dev_to_f64(t):
    """A bf16 or fp16 device tensor as float64 numpy values (exact)."""
    return t.cpu().float().numpy().astype(np.float64)


def run(moe, x, logits, **kw):
    ids, gates, perm, offsets = moe.plan(logits)
    out = torch.empty((x.shape[0], moe.H), dtype=moe.dtype, device=x.device)
    hm.hmoe_forward(moe.layer, x, ids, gates, perm, offsets, out, moe.ws, **kw)
    torch.cuda.synchronize()
    hm.hmoe_check_device_status(moe.ws)
    return out, (ids, gates, perm, offsets)


def oracle_out(L, x, ids, gates, tokens=None, cols=None):
    xf = x.float().cpu().numpy().astype(np.float64)
    return olayer.moe_forward(xf, ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64), L.expert_numpy,
                              L.H, L.I, tokens=tokens, cols=cols)


def oracle_rows(L, x, ids, gates, tokens=None):
    """oracle_out over all columns, with the per-expert steps spread over host processes
    (tests/oracle_pool.py): for tests that reach many experts of a full-size layer."""
    xf = x.float().cpu().numpy().astype(np.float64)
    return oracle_pool.moe_rows(xf, ids.cpu().numpy(), gates.cpu().numpy().astype(np.float64), L.expert_numpy,
                                L.H, L.I, tokens=tokens)


def cover_tokens(ids, perm, offsets, stride=0):
    """Tokens that reach every routed expert: for each expert, the token of its first and of
    its last routed slot (so each expert's first and last, possibly ragged, token tile is
    checked), plus every stride-th token if stride > 0. Sorted, unique."""
    ids = ids.cpu().numpy()
    perm = perm.cpu().numpy()
    off = offsets.cpu().numpy()
    k = ids.shape[1]
    toks = set()
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            toks.add(int(perm[off[e]]) // k)
            toks.add(int(perm[off[e + 1] - 1]) // k)
    if stride > 0:
        toks.update(range(0, ids.shape[0], stride))
    return sorted(toks)


def assert_rows_close(got, ref, tol=REL_TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref).max(axis=1)
    scale = np.abs(ref).max(axis=1)
    worst = float((err / np.maximum(scale, 1e-30)).max()) if len(err) else 0.0
    assert np.all(err <= tol * scale), f"row-relative error {worst:.3e} > {tol}"
    return worst


def layer_on(device, **kw):
    return synth.make_layer(device=device, **kw)
