"""nf3_moe_gb300 -- the hybrid W4A16 mixture-of-experts layer on GB300 (sm_103a).

This is the Python face of libhmoe, the C ABI declared in include/hmoe.h.
The functions keep the C names and take torch tensors. PyTorch supplies
only device memory and streams. Every step of the layer runs in the
library's CUDA kernels.

Typical use (see ``HybridMoELayer`` for the same thing with owned buffers):

    layer = hmoe_pack_weights(desc, bit_map, experts, kept_buf, nf3_buf)
    hmoe_workspace_init(ws)
    hmoe_plan_routes(layer, logits, ids, gates, perm, offsets, ws)
    hmoe_forward(layer, x, ids, gates, perm, offsets, out, ws)
"""

import ctypes

import torch

from . import _lib
from ._lib import (FMT_MXFP4, FMT_NF3, FMT_NVFP4, PATH_AUTO, PATH_GROUPED, PATH_STREAM,  # noqa: F401
                   TIERS_KEPT_FIRST, TIERS_NF3_FIRST, TIERS_ONE_LAUNCH, HmoeError, LayerDesc, LinearDesc,
                   DEBUG_NO_COPIES, DEBUG_GROUPED_PAIR, ACT_BF16, ACT_F16, ACT_QUANT_NONE, ACT_QUANT_NVFP4)

__all__ = [
    "LayerDesc", "HmoeError", "hmoe_packed_size", "hmoe_workspace_size", "hmoe_workspace_init",
    "hmoe_pack_weights", "hmoe_plan_routes", "hmoe_forward", "hmoe_check_device_status",
    "hmoe_debug_dequant", "hmoe_debug_decode_operand", "HybridMoELayer", "library_path",
    "LinearDesc", "hmoe_linear_packed_size", "hmoe_linear_workspace_size", "hmoe_linear_pack", "hmoe_linear_forward",
    "LinearW4A16", "ACT_BF16", "ACT_F16", "act_torch_dtype", "ACT_QUANT_NONE", "ACT_QUANT_NVFP4",
    "hmoe_quantize_act_nvfp4",
]


def library_path():
    return _lib.LIB_PATH


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _desc(H, I, E, topk, kept_format=FMT_NVFP4, act_dtype=ACT_BF16, act_globals=None):
    """act_globals: None (W4A16), or (g13, g2): W4A4 with those static activation global scales."""
    if act_globals is None:
        return LayerDesc(H, I, E, topk, kept_format, act_dtype, ACT_QUANT_NONE, 0.0, 0.0)
    return LayerDesc(H, I, E, topk, kept_format, act_dtype, ACT_QUANT_NVFP4, float(act_globals[0]),
                     float(act_globals[1]))


def act_torch_dtype(act_dtype):
    """The torch dtype of x, h and out for an ACT_* value."""
    return {ACT_BF16: torch.bfloat16, ACT_F16: torch.float16}[int(act_dtype)]


def _bitmap_arg(bit_map):
    if bit_map is None:
        return None, None
    arr = (ctypes.c_int8 * len(bit_map))(*[int(b) for b in bit_map])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


# ------------------------------------------------------------------ argument checks
# The library sees raw device pointers only, so the binding checks every tensor it hands over:
# type, dtype, shape (or, for checkpoint and packed buffers, size in bytes), layout and device.
# A tensor of the wrong shape would otherwise have the kernels read or write past its end.
# The checks run on the host before the library is called; each raises ValueError (TypeError
# for a non-tensor). cuda=False skips the device checks, so that the rest can be tested
# without a GPU.

def _nbytes(t):
    return t.numel() * t.element_size()


def _need(name, t, shape=None, dtype=None, min_bytes=None, device=None, cuda=True):
    """shape: a tuple whose None entries match any extent."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and (t.dim() != len(shape) or
                              any(w is not None and int(g) != int(w) for g, w in zip(t.shape, shape))):
        want = "[" + ", ".join("*" if w is None else str(int(w)) for w in shape) + "]"
        raise ValueError(f"{name} must have shape {want}, got {list(t.shape)}")
    if min_bytes is not None and _nbytes(t) < min_bytes:
        raise ValueError(f"{name} holds {_nbytes(t)} bytes; at least {min_bytes} are needed")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cuda:
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
        if device is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the other arguments on {device}")


def _matrix_bytes(fmt, N, K):
    """(codes bytes, scales bytes) of one [N, K] matrix in the logical layout of include/hmoe.h."""
    if fmt == FMT_NVFP4:
        return N * K // 2, N * K // 16
    if fmt == FMT_MXFP4:
        return N * K // 2, N * K // 32
    return N * K * 3 // 8, N * (K // 64) * 2


def _check_route_bufs(desc, T, ids, gates, perm, offsets, device, cuda):
    k, E = int(desc.topk), int(desc.E)
    _need("ids", ids, (T, k), torch.int32, device=device, cuda=cuda)
    _need("gates", gates, (T, k), torch.float32, device=device, cuda=cuda)
    _need("perm", perm, (T * k,), torch.int32, device=device, cuda=cuda)
    _need("offsets", offsets, (E + 1,), torch.int32, device=device, cuda=cuda)


def _check_plan(desc, logits, ids, gates, perm, offsets, ws, cuda=True):
    _need("logits", logits, (None, int(desc.E)), torch.float32, cuda=cuda)
    _check_route_bufs(desc, logits.shape[0], ids, gates, perm, offsets, logits.device, cuda)
    _need("ws", ws, device=logits.device, cuda=cuda)


def _check_forward(desc, x, ids, gates, perm, offsets, out, ws, cuda=True):
    """ws None: the static entry point, which takes no workspace."""
    dt, H = act_torch_dtype(desc.act_dtype), int(desc.H)
    _need("x", x, (None, H), dt, cuda=cuda)
    T = x.shape[0]
    _check_route_bufs(desc, T, ids, gates, perm, offsets, x.device, cuda)
    _need("out", out, (T, H), dt, device=x.device, cuda=cuda)
    if ws is not None:
        _need("ws", ws, device=x.device, cuda=cuda)


def _check_pack(desc, bit_map, experts, kept_buf, nf3_buf, cuda=True):
    kb, nb = hmoe_packed_size(desc, bit_map)          # the descriptor and bit map checks (library)
    E, H, I = int(desc.E), int(desc.H), int(desc.I)
    if len(experts) != E:
        raise ValueError(f"expected {E} experts, got {len(experts)}")
    for e, (c13, s13, _, c2, s2, _) in enumerate(experts):
        fmt = FMT_NF3 if bit_map is not None and int(bit_map[e]) == 3 else int(desc.kept_format)
        for nm, (N, K), c, sc in (("W13", (2 * I, H), c13, s13), ("W2", (H, I), c2, s2)):
            cb, sb = _matrix_bytes(fmt, N, K)
            _need(f"expert {e} {nm} codes", c, min_bytes=cb, cuda=cuda)
            _need(f"expert {e} {nm} scales", sc, min_bytes=sb, cuda=cuda)
    if kb:
        _need("kept_buf", kept_buf, min_bytes=kb, cuda=cuda)
    if nb:
        _need("nf3_buf", nf3_buf, min_bytes=nb, cuda=cuda)


def _check_linear_forward(desc, x, out, ws, cuda=True):
    dt = act_torch_dtype(desc.act_dtype)
    _need("x", x, (None, int(desc.K)), dt, cuda=cuda)
    _need("out", out, (x.shape[0], int(desc.N)), dt, device=x.device, cuda=cuda)
    _need("ws", ws, device=x.device, cuda=cuda)


def hmoe_packed_size(desc, bit_map=None):
    kb, nb = ctypes.c_size_t(), ctypes.c_size_t()
    keep, bm = _bitmap_arg(bit_map)
    _lib.check(_lib.lib().hmoe_packed_size(ctypes.byref(desc), bm, ctypes.byref(kb), ctypes.byref(nb)))
    return kb.value, nb.value


def hmoe_workspace_size(desc, max_tokens):
    b = ctypes.c_size_t()
    _lib.check(_lib.lib().hmoe_workspace_size(ctypes.byref(desc), int(max_tokens), ctypes.byref(b)))
    return b.value


def hmoe_auto_path(desc, T):
    """PATH_STREAM or PATH_GROUPED: the path hmoe_forward takes for T tokens with path=PATH_AUTO."""
    out = ctypes.c_int()
    _lib.check(_lib.lib().hmoe_auto_path(ctypes.byref(desc), int(T), ctypes.byref(out)))
    return out.value


def hmoe_workspace_init(ws, stream=None):
    _lib.check(_lib.lib().hmoe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


class Layer:
    """Owns the C handle. It keeps the tier buffers alive while it lives."""

    def __init__(self, handle, desc, kept_buf, nf3_buf):
        self.handle = handle
        self.desc = desc
        self.kept_buf, self.nf3_buf = kept_buf, nf3_buf

    def expert_info(self, e):
        f, a, b = ctypes.c_int(), ctypes.c_float(), ctypes.c_float()
        _lib.check(_lib.lib().hmoe_layer_expert_info(self.handle, int(e), ctypes.byref(f), ctypes.byref(a),
                                                     ctypes.byref(b)))
        return f.value, a.value, b.value

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib._LIB is not None:
            _lib._LIB.hmoe_layer_destroy(h)


def hmoe_pack_weights(desc, bit_map, experts, kept_buf, nf3_buf, stream=None):
    """experts: list of E tuples (w13_codes, w13_scales, w13_global, w2_codes, w2_scales, w2_global).
    Tensors must be CUDA tensors in the logical layout of include/hmoe.h."""
    E = desc.E
    _check_pack(desc, bit_map, experts, kept_buf, nf3_buf)
    src = (_lib.ExpertSrc * E)()
    for e, (c13, s13, g13, c2, s2, g2) in enumerate(experts):
        src[e] = _lib.ExpertSrc(c13.data_ptr(), s13.data_ptr(), float(g13), c2.data_ptr(), s2.data_ptr(), float(g2))
    keep, bm = _bitmap_arg(bit_map)
    h = ctypes.c_void_p()
    _lib.check(_lib.lib().hmoe_pack_weights(ctypes.byref(desc), bm, src, _ptr(kept_buf), _ptr(nf3_buf),
                                            _stream(stream), ctypes.byref(h)))
    return Layer(h, desc, kept_buf, nf3_buf)


def hmoe_plan_routes(layer, logits, ids, gates, perm, offsets, ws, stream=None):
    _check_plan(layer.desc, logits, ids, gates, perm, offsets, ws)
    T = logits.shape[0]
    _lib.check(_lib.lib().hmoe_plan_routes(layer.handle, _ptr(logits), T, _ptr(ids), _ptr(gates), _ptr(perm),
                                           _ptr(offsets), _ptr(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)))


def hmoe_forward(layer, x, ids, gates, perm, offsets, out, ws, stream=None, tier_order=TIERS_ONE_LAUNCH,
                 path=PATH_AUTO, wait_limit_us=0, debug_flags=0, stage_events=None):
    """stage_events: optional list of recorded torch.cuda.Event (up to 4); see hmoe_forward_opts."""
    _check_forward(layer.desc, x, ids, gates, perm, offsets, out, ws)
    T = x.shape[0]
    evs, n_ev = None, 0
    if stage_events:
        arr = (ctypes.c_void_p * len(stage_events))(*[ctypes.c_void_p(e.cuda_event) for e in stage_events])
        evs, n_ev = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), len(stage_events)
    opts = _lib.ForwardOpts(int(tier_order), int(path), int(wait_limit_us), int(debug_flags), evs, n_ev)
    _lib.check(_lib.lib().hmoe_forward_ex(layer.handle, _ptr(x), T, _ptr(ids), _ptr(gates), _ptr(perm),
                                          _ptr(offsets), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                          ctypes.byref(opts), _stream(stream)))


def hmoe_launch_count():
    return int(_lib.lib().hmoe_launch_count())


def hmoe_check_device_status(ws, stream=None):
    _lib.check(_lib.lib().hmoe_check_device_status(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def _debug_shape(desc, which):
    """[N, K] of the matrix which (13 or 2) selects; None for another value (the library rejects it)."""
    H, I = int(desc.H), int(desc.I)
    return {13: (2 * I, H), 2: (H, I)}.get(int(which))


def hmoe_debug_dequant(layer, expert, which, dst, stream=None):
    shape = _debug_shape(layer.desc, which)
    if shape is not None:
        _need("dst", dst, shape, act_torch_dtype(layer.desc.act_dtype))
    _lib.check(_lib.lib().hmoe_debug_dequant(layer.handle, int(expert), int(which), _ptr(dst), _stream(stream)))


def hmoe_debug_decode_operand(layer, expert, which, dst, scales, stream=None):
    """The weight-streaming kernel's operand (dst [N, K] of the activation type) and per-64-group
    factors (scales fp32 [N, K/64])."""
    shape = _debug_shape(layer.desc, which)
    if shape is not None:
        _need("dst", dst, shape, act_torch_dtype(layer.desc.act_dtype))
        _need("scales", scales, (shape[0], shape[1] // 64), torch.float32, device=dst.device)
    _lib.check(_lib.lib().hmoe_debug_decode_operand(layer.handle, int(expert), int(which), _ptr(dst), _ptr(scales),
                                                    _stream(stream)))


class HybridMoELayer:
    """One hybrid MoE layer with its packed tier buffers and workspace owned as torch tensors.

    desc_args: H, I, E, topk, kept_format, act_dtype, act_globals (None for
    W4A16, (g13, g2) for W4A4). bit_map: per-expert 4/3 list, or None for
    uniform. experts: as in hmoe_pack_weights. max_tokens sizes the
    workspace.
    """

    def __init__(self, H, I, E, topk, bit_map, experts, kept_format=FMT_NVFP4, max_tokens=8, device="cuda",
                 act_dtype=ACT_BF16, act_globals=None):
        self.desc = _desc(H, I, E, topk, kept_format, act_dtype, act_globals)
        self.dtype = act_torch_dtype(act_dtype)
        kb, nb = hmoe_packed_size(self.desc, bit_map)
        self.kept_buf = torch.empty(max(kb, 16), dtype=torch.uint8, device=device) if kb else None
        self.nf3_buf = torch.empty(max(nb, 16), dtype=torch.uint8, device=device) if nb else None
        self.layer = hmoe_pack_weights(self.desc, bit_map, experts, self.kept_buf, self.nf3_buf)
        self.max_tokens = max_tokens
        self.ws = torch.empty(hmoe_workspace_size(self.desc, max_tokens), dtype=torch.uint8, device=device)
        hmoe_workspace_init(self.ws)
        self.topk = topk
        self.E = E
        self.H = H

    def plan(self, logits):
        T = logits.shape[0]
        dev = logits.device
        ids = torch.empty((T, self.topk), dtype=torch.int32, device=dev)
        gates = torch.empty((T, self.topk), dtype=torch.float32, device=dev)
        perm = torch.empty((T * self.topk,), dtype=torch.int32, device=dev)
        offsets = torch.empty((self.E + 1,), dtype=torch.int32, device=dev)
        hmoe_plan_routes(self.layer, logits, ids, gates, perm, offsets, self.ws)
        return ids, gates, perm, offsets

    def __call__(self, x, logits, tier_order=TIERS_ONE_LAUNCH, path=PATH_AUTO, out=None):
        ids, gates, perm, offsets = self.plan(logits)
        if out is None:
            out = torch.empty((x.shape[0], self.H), dtype=self.dtype, device=x.device)
        hmoe_forward(self.layer, x, ids, gates, perm, offsets, out, self.ws, tier_order=tier_order, path=path)
        return out


def hmoe_forward_static(layer, x, ids, gates, perm, offsets, out, stream=None):
    """hmoe_forward without a caller workspace (see include/hmoe.h): the scratch is a fixed
    per-device array inside the library, so the call allocates no device memory."""
    _check_forward(layer.desc, x, ids, gates, perm, offsets, out, None)
    T = x.shape[0]
    _lib.check(_lib.lib().hmoe_forward_static(layer.handle, _ptr(x), T, _ptr(ids), _ptr(gates), _ptr(perm),
                                              _ptr(offsets), _ptr(out), _stream(stream)))


def hmoe_check_device_status_static(stream=None):
    _lib.check(_lib.lib().hmoe_check_device_status_static(_stream(stream)))


# ------------------------------------------------------------------ dense Linear W4A16
def hmoe_linear_packed_size(desc):
    b = ctypes.c_size_t()
    _lib.check(_lib.lib().hmoe_linear_packed_size(ctypes.byref(desc), ctypes.byref(b)))
    return b.value


def hmoe_linear_workspace_size(desc, max_tokens):
    b = ctypes.c_size_t()
    _lib.check(_lib.lib().hmoe_linear_workspace_size(ctypes.byref(desc), int(max_tokens), ctypes.byref(b)))
    return b.value


class Linear:
    """Owns the C handle of a packed dense W4A16 matrix; keeps the packed buffer alive."""

    def __init__(self, handle, desc, packed):
        self.handle, self.desc, self.packed = handle, desc, packed

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib._LIB is not None:
            _lib._LIB.hmoe_linear_destroy(h)


def hmoe_linear_pack(desc, codes, scales, global_scale, packed, stream=None):
    nbytes = hmoe_linear_packed_size(desc)            # the descriptor checks (library)
    cb, sb = _matrix_bytes(int(desc.fmt), int(desc.N), int(desc.K))
    _need("codes", codes, min_bytes=cb)
    _need("scales", scales, min_bytes=sb, device=codes.device)
    _need("packed", packed, min_bytes=nbytes, device=codes.device)
    h = ctypes.c_void_p()
    _lib.check(_lib.lib().hmoe_linear_pack(ctypes.byref(desc), _ptr(codes), _ptr(scales), float(global_scale),
                                           _ptr(packed), _stream(stream), ctypes.byref(h)))
    return Linear(h, desc, packed)


def hmoe_linear_forward(linear, x, out, ws, stream=None, path=PATH_AUTO, wait_limit_us=0, debug_flags=0):
    _check_linear_forward(linear.desc, x, out, ws)
    opts = _lib.ForwardOpts(TIERS_ONE_LAUNCH, int(path), int(wait_limit_us), int(debug_flags), None, 0)
    _lib.check(_lib.lib().hmoe_linear_forward_ex(linear.handle, _ptr(x), int(x.shape[0]), _ptr(out), _ptr(ws),
                                                 ws.numel() * ws.element_size(), ctypes.byref(opts), _stream(stream)))


class LinearW4A16:
    """A dense W4A16 Linear with its packed matrix and workspace owned as torch tensors.

    codes, scales: CUDA tensors of one [N, K] matrix in the logical layout of fmt
    (include/hmoe.h); global_scale: the NVFP4 global scale (ignored otherwise).
    """

    def __init__(self, N, K, fmt, codes, scales, global_scale=1.0, max_tokens=8, device="cuda", act_dtype=ACT_BF16):
        self.desc = LinearDesc(N, K, fmt, act_dtype)
        self.dtype = act_torch_dtype(act_dtype)
        self.packed = torch.empty(hmoe_linear_packed_size(self.desc), dtype=torch.uint8, device=device)
        self.linear = hmoe_linear_pack(self.desc, codes, scales, global_scale, self.packed)
        self.ws = torch.empty(hmoe_linear_workspace_size(self.desc, max_tokens), dtype=torch.uint8, device=device)
        hmoe_workspace_init(self.ws)
        self.N = N

    def __call__(self, x, out=None, path=PATH_AUTO):
        if out is None:
            out = torch.empty((x.shape[0], self.N), dtype=self.dtype, device=x.device)
        hmoe_linear_forward(self.linear, x, out, self.ws, path=path)
        return out


def hmoe_quantize_act_nvfp4(x, global_scale, codes, scales, stream=None):
    """NVFP4 activation quantisation of x [rows, K] (bf16 or fp16): codes uint8 [rows, K/2],
    scales uint8 [rows, K/16] (include/hmoe.h)."""
    _need("x", x, (None, None))
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"x must be torch.bfloat16 or torch.float16, got {x.dtype}")
    R, K = x.shape
    if K % 16 == 0:                                  # other K: the library rejects the call
        _need("codes", codes, (R, K // 2), torch.uint8, device=x.device)
        _need("scales", scales, (R, K // 16), torch.uint8, device=x.device)
    act = ACT_F16 if x.dtype == torch.float16 else ACT_BF16
    _lib.check(_lib.lib().hmoe_quantize_act_nvfp4(_ptr(x), int(x.shape[0]), int(x.shape[1]), act,
                                                  ctypes.c_float(global_scale), _ptr(codes), _ptr(scales),
                                                  _stream(stream)))
