"""CPU tests of the C ABI surface: the library loads, exports every symbol include/hmoe.h
declares, and validates arguments on the host (no compute call needs a GPU here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from nf3_moe_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "hmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hmoe_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    from nf3_moe_gb300 import _lib
    declared = _declared()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(_lib.EXPORTS)


def _prototypes():
    """{name: (return type text, [parameter texts])} of every function include/hmoe.h declares."""
    src = open(os.path.join(ROOT, "include", "hmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w \*]*?)\s*\b(hmoe_[a-z_0-9]+)\s*\(([^;{)]*)\)\s*;", src):
        params = " ".join(params.split())
        out[name] = (ret.split()[-1] if ret.split() else ret, [] if params in ("", "void") else params.split(", "))
    return out


def _ctype_kind(c):
    if c is None:
        return "void"
    if c in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(c, ctypes._Pointer):
        return "ptr"
    # c_size_t and c_uint64 are one class on LP64 platforms: both are "u64"
    return {ctypes.c_int: "int", ctypes.c_size_t: "u64", ctypes.c_float: "float", ctypes.c_uint64: "u64"}[c]


def _c_kind(text):
    if "*" in text or text.split()[0] == "hmoe_stream_t":
        return "ptr"
    base = text.replace("const ", "").split()[0]
    return {"int": "int", "size_t": "u64", "float": "float", "hmoe_status": "int", "uint64_t": "u64",
            "void": "void"}[base]


def test_binding_signatures_match_the_header(lib):
    """Every ctypes prototype has the header's parameter count and, per parameter, the same kind
    (pointer, int, 64-bit unsigned, float): a mismatch would pass garbage across the ABI silently."""
    protos = _prototypes()
    assert set(protos) == set(_declared())
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert len(fn.argtypes) == len(params), (name, params)
        for a, p in zip(fn.argtypes, params):
            assert _ctype_kind(a) == _c_kind(p), (name, p, a)
        want_ret = "ptr" if ret.endswith("*") else _c_kind(ret)
        assert _ctype_kind(fn.restype) == want_ret, (name, ret, fn.restype)


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "hmoe.h"

int main(void) {
  hmoe_layer_desc d;
  size_t kept = 0, nf3 = 0, ws = 0;
  int path = -1, e;
  int8_t bit_map[256];
  memset(&d, 0, sizeof d);                      /* a zeroed descriptor: bf16, W4A16 */
  d.H = 6144; d.I = 2048; d.E = 256; d.topk = 8; d.kept_format = HMOE_FMT_NVFP4;
  for (e = 0; e < 256; ++e) bit_map[e] = (int8_t)(e < 64 ? 4 : 3);
  if (hmoe_packed_size(&d, bit_map, &kept, &nf3) != HMOE_OK) return 1;
  if (hmoe_workspace_size(&d, 4096, &ws) != HMOE_OK) return 2;
  if (hmoe_auto_path(&d, 4096, &path) != HMOE_OK) return 3;
  if (hmoe_plan_routes(NULL, NULL, 1, NULL, NULL, NULL, NULL, NULL, 0, NULL) != HMOE_ERR_INVALID_ARG) return 4;
  if (strlen(hmoe_last_error()) == 0) return 5;
  printf("%d %zu %zu %zu %d\n", hmoe_version(), kept, nf3, ws, path);
  return 0;
}
"""


def test_header_is_plain_c_and_links_from_c(lib, tmp_path):
    """A C99 client, compiled with -Wall -Werror -pedantic against include/hmoe.h and linked
    with libhmoe.so, calls the host-only entry points: the boundary needs no C++ and no torch."""
    import shutil
    import subprocess
    import nf3_moe_gb300 as hm
    from nf3_moe_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(_lib.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), f"-L{libdir}", "-l:libhmoe.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    version, kept, nf3, ws, path = (int(v) for v in r.stdout.split())
    d = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4)
    assert version == lib.hmoe_version()
    assert (kept, nf3) == hm.hmoe_packed_size(d, [4] * 64 + [3] * 192)
    assert ws == hm.hmoe_workspace_size(d, 4096)
    assert path == hm.PATH_GROUPED


def test_version_and_last_error(lib):
    assert lib.hmoe_version() >= 100
    assert isinstance(lib.hmoe_last_error(), bytes)


def test_host_validation_without_gpu(lib):
    import nf3_moe_gb300 as hm
    d = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4)
    kept, nf3 = hm.hmoe_packed_size(d, [4] * 64 + [3] * 192)
    assert kept == 64 * 21_233_664 and nf3 == 192 * 15_335_424
    dm = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_MXFP4)
    assert hm.hmoe_packed_size(dm, [4] * 64 + [3] * 192)[0] == 64 * 20_054_016
    assert hm.hmoe_packed_size(hm.LayerDesc(2048, 768, 128, 8, 4), None) == (128 * 2_654_208, 0)
    sizes = [hm.hmoe_workspace_size(d, t) for t in (0, 1, 8, 9, 4096)]
    assert sizes == sorted(sizes)
    # fp16 layers: same packed sizes and workspace (2-byte activations either way)
    d16 = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4, hm.ACT_F16)
    assert hm.hmoe_packed_size(d16, [4] * 64 + [3] * 192) == (kept, nf3)
    assert [hm.hmoe_workspace_size(d16, t) for t in (0, 1, 8, 9, 4096)] == sizes
    for bad, status in [(hm.LayerDesc(6144, 2048, 256, 8, 7), -1), (hm.LayerDesc(6100, 2048, 256, 8, 4), -2),
                        (hm.LayerDesc(6144, 2000, 256, 8, 4), -2), (hm.LayerDesc(6144, 2048, 600, 8, 4), -2),
                        (hm.LayerDesc(6144, 2048, 4, 8, 4), -2), (hm.LayerDesc(0, 2048, 4, 2, 4), -1),
                        (hm.LayerDesc(6144, 2048, 256, 8, 4, 2), -1), (hm.LayerDesc(6144, 2048, 256, 8, 4, -1), -1)]:
        with pytest.raises(hm.HmoeError) as ei:
            hm.hmoe_workspace_size(bad, 8)
        assert ei.value.status == status
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_packed_size(d, [4] * 255 + [2])
    assert ei.value.status == -4
    # slots are 32-bit indices: T * topk may reach INT_MAX but not pass it
    d1 = hm.LayerDesc(256, 128, 8, 1, hm.FMT_NVFP4)
    assert hm.hmoe_workspace_size(d1, 2**31 - 1) > 0
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_workspace_size(d, 2**31 // 8)
    assert ei.value.status == -2


def test_auto_path_rule():
    """Streaming while T * topk <= 8 * E, grouped above; every T <= 8 streams."""
    import nf3_moe_gb300 as hm
    hyb = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4)
    uni = hm.LayerDesc(2048, 768, 128, 8, hm.FMT_NVFP4)
    tiny = hm.LayerDesc(256, 128, 8, 2, hm.FMT_NVFP4)
    S, G = hm.PATH_STREAM, hm.PATH_GROUPED
    cases = [(hyb, 0, S), (hyb, 1, S), (hyb, 8, S), (hyb, 64, S), (hyb, 256, S), (hyb, 257, G), (hyb, 4096, G),
             (uni, 128, S), (uni, 129, G), (tiny, 8, S), (tiny, 32, S), (tiny, 33, G), (tiny, 37, G)]
    for desc, T, want in cases:
        assert hm.hmoe_auto_path(desc, T) == want, (desc.E, T)
    # a layer whose top-k exceeds 8 * E / T for every T > 8 still streams at T <= 8
    assert hm.hmoe_auto_path(hm.LayerDesc(256, 128, 8, 8, hm.FMT_NVFP4), 8) == S
    with pytest.raises(hm.HmoeError) as ei:
        hm.hmoe_auto_path(hyb, -1)
    assert ei.value.status == -1


def test_null_handles_rejected(lib):
    assert lib.hmoe_plan_routes(None, None, 1, None, None, None, None, None, 0, None) == -1
    assert lib.hmoe_forward(None, None, 1, None, None, None, None, None, None, 0, None) == -1
    assert lib.hmoe_debug_dequant(None, 0, 13, None, None) == -1
    assert lib.hmoe_check_device_status(None, 0, None) == -1
    desc = __import__("nf3_moe_gb300")._lib.LayerDesc(256, 128, 8, 2, 4)
    h = ctypes.c_void_p()
    assert lib.hmoe_pack_weights(ctypes.byref(desc), None, None, None, None, None, ctypes.byref(h)) == -1
    assert b"NULL" in lib.hmoe_last_error()
    lib.hmoe_layer_destroy(None)


def test_linear_desc_checks_on_host(lib):
    import nf3_moe_gb300 as hm
    assert hm.hmoe_linear_packed_size(hm.LinearDesc(256, 384, hm.FMT_NF3)) == 2 * 6 * 3328
    assert hm.hmoe_linear_packed_size(hm.LinearDesc(128, 64, hm.FMT_NVFP4)) == 4608
    assert hm.hmoe_linear_packed_size(hm.LinearDesc(128, 64, hm.FMT_NVFP4, hm.ACT_F16)) == 4608
    for bad, status in (((100, 64, 4), -2), ((128, 32, 4), -2), ((128, 64, 7), -1), ((0, 64, 3), -1),
                        ((128, 64, 4, 3), -1)):
        with pytest.raises(hm.HmoeError) as ei:
            hm.hmoe_linear_packed_size(hm.LinearDesc(*bad))
        assert ei.value.status == status
    assert hm.hmoe_linear_workspace_size(hm.LinearDesc(256, 384, hm.FMT_NVFP4), 0) == 768


def test_w4a4_desc_and_quantizer_checks_on_host(lib):
    import nf3_moe_gb300 as hm
    base = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4)
    w4 = hm.LayerDesc(6144, 2048, 256, 8, hm.FMT_NVFP4, hm.ACT_BF16, hm.ACT_QUANT_NVFP4, 1e-3, 2e-3)
    # the W4A4 workspace holds the quantised input [T][H] on top
    assert hm.hmoe_workspace_size(w4, 64) - hm.hmoe_workspace_size(base, 64) == 64 * 6144 * 2
    for bad in (hm.LayerDesc(6144, 2048, 256, 8, 4, 0, 2, 1e-3, 1e-3), hm.LayerDesc(6144, 2048, 256, 8, 4, 0, 1, 0.0, 1e-3),
                hm.LayerDesc(6144, 2048, 256, 8, 4, 0, 1, 1e-3, float("inf"))):
        with pytest.raises(hm.HmoeError) as ei:
            hm.hmoe_workspace_size(bad, 8)
        assert ei.value.status == -1
    q = lib.hmoe_quantize_act_nvfp4
    assert q(None, 0, 256, 0, ctypes.c_float(1e-3), None, None, None) == 0    # rows = 0: nothing to do
    assert q(None, -1, 256, 0, ctypes.c_float(1e-3), None, None, None) == -1
    assert q(None, 1, 250, 0, ctypes.c_float(1e-3), None, None, None) == -1
    assert q(None, 1, 256, 7, ctypes.c_float(1e-3), None, None, None) == -1
    assert q(None, 1, 256, 0, ctypes.c_float(-1.0), None, None, None) == -1
    assert q(None, 1, 256, 0, ctypes.c_float(1e-3), None, None, None) == -1  # NULL buffers
