"""The dense-Linear W4A16 entry points against oracle.linear, on both paths.

Tolerance as for the layer: per output row, max|out - ref| <= 2e-2 * max|ref|
(fp32 accumulation, bf16 result).
"""

import numpy as np
import pytest
import torch

import nf3_moe_gb300 as hm
import synth
from oracle import linear as olinear
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _matrix(fmt, N, K, seed=0):
    w = synth.gen_master(seed, 2, N, K, seed=seed, device="cuda")
    return synth.quantise(fmt, w)


def _ref(x, fmt, codes, scales, g, K):
    c = codes.cpu().numpy()
    s = scales.cpu().numpy()
    if fmt == synth.FMT_NF3:
        s = s.view(np.uint16)
    return olinear.linear_forward(x.float().cpu().numpy().astype(np.float64), fmt, c, s, g, K)


@pytest.mark.parametrize("fmt", [synth.FMT_NVFP4, synth.FMT_MXFP4, synth.FMT_NF3])
def test_linear_small_all_formats_both_paths(fmt):
    N, K = 256, 384
    codes, scales, g = _matrix(fmt, N, K, seed=3)
    lin = hm.LinearW4A16(N, K, fmt, codes, scales, g, max_tokens=300)
    for T in (1, 5, 8, 9, 64, 300):
        x = synth.gen_x(T, K, seed=T, device="cuda")
        ref = _ref(x, fmt, codes, scales, g, K)
        auto = lin(x)
        torch.cuda.synchronize()
        hm.hmoe_check_device_status(lin.ws)
        U.assert_rows_close(auto.float().cpu().numpy(), ref)
        other_path = hm.PATH_GROUPED if T <= 8 else hm.PATH_STREAM
        other = lin(x, path=other_path)
        torch.cuda.synchronize()
        hm.hmoe_check_device_status(lin.ws)
        U.assert_rows_close(other.float().cpu().numpy(), ref)


@pytest.mark.parametrize("fmt,N,K", [(synth.FMT_NVFP4, 6144, 2048), (synth.FMT_NF3, 4096, 6144)])
def test_linear_full_size(fmt, N, K):
    """Matrices of the 256-expert layer's shapes (W2 as [H, I], W13 as [2I, H]) at decode and
    prefill sizes; every row checked against the oracle."""
    codes, scales, g = _matrix(fmt, N, K, seed=11)
    lin = hm.LinearW4A16(N, K, fmt, codes, scales, g, max_tokens=1024)
    for T in (8, 1024):
        x = synth.gen_x(T, K, seed=T + 1, device="cuda")
        out = lin(x)
        torch.cuda.synchronize()
        hm.hmoe_check_device_status(lin.ws)
        U.assert_rows_close(out.float().cpu().numpy(), _ref(x, fmt, codes, scales, g, K))


def test_linear_zero_tokens_and_bad_arguments():
    N, K = 128, 64
    codes, scales, g = _matrix(synth.FMT_NVFP4, N, K)
    lin = hm.LinearW4A16(N, K, synth.FMT_NVFP4, codes, scales, g, max_tokens=4)
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    hm.hmoe_linear_forward(lin.linear, x, out, lin.ws)
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_linear_forward(lin.linear, synth.gen_x(5, K, device="cuda"),
                               torch.empty((5, N), dtype=torch.bfloat16, device="cuda"), lin.ws)
    assert ei.value.status == -3                       # workspace sized for 4 rows
