"""Python binding of the GB300 latent mixture-of-experts layer (``liblmoe.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Functions carry the C names of ``include/lmoe.h`` and take torch
CUDA tensors (device memory and the current stream come from PyTorch).  There
is no CPU fallback: if the library is missing or cannot load, importing the
binding raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH
from ._build import build, up_to_date

__all__ = [
    "LmoeDims", "LmoeWeights", "LmoeWsLayout", "LmoeError", "build", "load",
    "lmoe_workspace_bytes", "lmoe_workspace_layout", "lmoe_route", "lmoe_route_noalloc", "lmoe_pool", "lmoe_experts_mxfp4",
    "lmoe_norm_combine_unpool", "lmoe_forward", "lmoe_forward_host", "lmoe_host_workspace_bytes", "lmoe_forward_routed",
    "lmoe_block_workspace_bytes",
    "lmoe_block_forward", "norms_of", "lmoe_experts_nvfp4", "lmoe_forward_nvfp4", "nvfp4_of",
    "lmoe_status_check", "lmoe_error_string",
    "lmoe_last_launch_count", "lmoe_selftest_e2m1", "lmoe_selftest_timeout", "lmoe_profile_events", "dims_of",
    "weights_of",
]

LMOE_OK, LMOE_EINVAL, LMOE_EUNSUPPORTED, LMOE_ECUDA, LMOE_ETIMEOUT, LMOE_EDEVICE_CHECK, LMOE_EWORKSPACE = \
    0, -1, -2, -3, -4, -5, -6
LMOE_ENOSCRATCH = -7


class LmoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("hidden", ctypes.c_int32), ("latent", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("eps", ctypes.c_float)]


class LmoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("router_w", "router_bias", "pooler_w", "w13_q", "w13_s", "w2_q",
                                               "w2_s", "norm_g", "unpooler_w")]


class LmoeBlockNorms(ctypes.Structure):
    _fields_ = [("pre_g", ctypes.c_void_p), ("post_g", ctypes.c_void_p), ("eps", ctypes.c_float)]


class LmoeNvfp4Scales(ctypes.Structure):
    _fields_ = [("w13_gs", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p)]


class LmoeWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "topk_idx", "topk_w", "expert_offsets", "sorted_rows",
                                               "row_pos", "x_lat", "y", "z", "total")]


class LmoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {lmoe_error_string(code)} ({code})")
        self.code = code


_lib = None


def load(path: str | None = None):
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"liblmoe.so is not built ({path}); run latent_moe_layer_fp32_gb300.build() "
                          "or __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    vp, sz, i32, dp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(LmoeDims)
    lib.lmoe_workspace_bytes.argtypes = [dp]
    lib.lmoe_workspace_bytes.restype = sz
    lib.lmoe_workspace_layout.argtypes = [dp, ctypes.POINTER(LmoeWsLayout)]
    lib.lmoe_route.argtypes = [dp] + [vp] * 8 + [vp, sz, vp]
    lib.lmoe_pool.argtypes = [dp, vp, vp, vp, vp, sz, vp]
    lib.lmoe_experts_mxfp4.argtypes = [dp] + [vp] * 8 + [vp, sz, vp]
    lib.lmoe_experts_nvfp4.argtypes = [dp] + [vp] * 10 + [vp, sz, vp]
    lib.lmoe_forward_nvfp4.argtypes = [dp, ctypes.POINTER(LmoeWeights), ctypes.POINTER(LmoeNvfp4Scales), vp, vp, vp,
                                       sz, vp]
    lib.lmoe_norm_combine_unpool.argtypes = [dp] + [vp] * 6 + [vp, sz, vp]
    lib.lmoe_forward.argtypes = [dp, ctypes.POINTER(LmoeWeights), vp, vp, vp, sz, vp]
    lib.lmoe_forward_host.argtypes = [dp, ctypes.POINTER(LmoeWeights), vp, vp, vp, sz, vp]
    lib.lmoe_host_workspace_bytes.argtypes = [dp]
    lib.lmoe_host_workspace_bytes.restype = sz
    lib.lmoe_forward_routed.argtypes = [dp, ctypes.POINTER(LmoeWeights), vp, vp, vp, vp, vp, sz, vp]
    lib.lmoe_block_workspace_bytes.argtypes = [dp]
    lib.lmoe_block_workspace_bytes.restype = sz
    lib.lmoe_block_forward.argtypes = [dp, ctypes.POINTER(LmoeWeights), ctypes.POINTER(LmoeBlockNorms), vp, vp, vp,
                                       sz, vp]
    lib.lmoe_status_check.argtypes = [vp, vp]
    lib.lmoe_error_string.argtypes = [i32]
    lib.lmoe_error_string.restype = ctypes.c_char_p
    lib.lmoe_last_launch_count.argtypes = []
    lib.lmoe_selftest_e2m1.argtypes = [vp]
    lib.lmoe_selftest_timeout.argtypes = [vp, sz, ctypes.c_uint, vp]
    lib.lmoe_selftest_timeout.restype = i32
    lib.lmoe_selftest_dequant_bf16.argtypes = [vp, vp, i32, vp]
    lib.lmoe_profile_events.argtypes = [vp, i32]
    lib.lmoe_route_noalloc.argtypes = [dp] + [vp] * 8 + [vp]
    lib.lmoe_set_option.argtypes = [i32, i32]
    lib.lmoe_last_launch_name.argtypes = [i32]
    lib.lmoe_last_launch_name.restype = ctypes.c_char_p
    for f in ("lmoe_workspace_layout", "lmoe_route", "lmoe_pool", "lmoe_experts_mxfp4", "lmoe_norm_combine_unpool",
              "lmoe_forward", "lmoe_forward_routed", "lmoe_block_forward", "lmoe_forward_nvfp4", "lmoe_experts_nvfp4",
              "lmoe_status_check", "lmoe_last_launch_count", "lmoe_selftest_e2m1",
              "lmoe_profile_events", "lmoe_route_noalloc", "lmoe_set_option", "lmoe_selftest_dequant_bf16",
              "lmoe_forward_host"):
        getattr(lib, f).restype = i32
    _lib = lib
    return lib


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------

def _ptr(t, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype is not None and t.dtype not in dtype:
        raise TypeError(f"unexpected dtype {t.dtype}, want one of {dtype}")
    return ctypes.c_void_p(t.data_ptr())


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_U8 = (torch.uint8,)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != LMOE_OK:
        raise LmoeError(rc, what)


def dims_of(T, hidden, latent, inter, n_experts, top_k, eps=1e-6) -> LmoeDims:
    return LmoeDims(T, hidden, latent, inter, n_experts, top_k, eps)


def weights_of(w: dict) -> LmoeWeights:
    """LmoeWeights from a dict of device tensors (keys as in the struct)."""
    return LmoeWeights(
        _ptr(w["router_w"], _F32), _ptr(w.get("router_bias"), _F32), _ptr(w["pooler_w"], _BF16),
        _ptr(w["w13_q"], _U8), _ptr(w["w13_s"], _U8), _ptr(w["w2_q"], _U8), _ptr(w["w2_s"], _U8),
        _ptr(w["norm_g"], _BF16), _ptr(w["unpooler_w"], _BF16))


# ---------------------------------------------------------------------------------------------
# the C calls
# ---------------------------------------------------------------------------------------------

def lmoe_error_string(code: int) -> str:
    return load().lmoe_error_string(int(code)).decode()


def lmoe_workspace_bytes(dims: LmoeDims) -> int:
    return int(load().lmoe_workspace_bytes(ctypes.byref(dims)))


def lmoe_workspace_layout(dims: LmoeDims) -> LmoeWsLayout:
    out = LmoeWsLayout()
    _check(load().lmoe_workspace_layout(ctypes.byref(dims), ctypes.byref(out)), "lmoe_workspace_layout")
    return out


def lmoe_route(dims, x, router_w, router_bias, topk_idx, topk_w, expert_offsets, sorted_rows, row_pos, ws,
               stream=None):
    _check(load().lmoe_route(ctypes.byref(dims), _ptr(x, _BF16), _ptr(router_w, _F32), _ptr(router_bias, _F32),
                             _ptr(topk_idx, _I32), _ptr(topk_w, _F32), _ptr(expert_offsets, _I32),
                             _ptr(sorted_rows, _I32), _ptr(row_pos, _I32), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "lmoe_route")


def lmoe_route_noalloc(dims, x, router_w, router_bias, topk_idx, topk_w, expert_offsets, sorted_rows, row_pos,
                       stream=None):
    """lmoe_route without a workspace (fixed library-owned scratch, T <= 64)."""
    _check(load().lmoe_route_noalloc(ctypes.byref(dims), _ptr(x, _BF16), _ptr(router_w, _F32),
                                     _ptr(router_bias, _F32), _ptr(topk_idx, _I32), _ptr(topk_w, _F32),
                                     _ptr(expert_offsets, _I32), _ptr(sorted_rows, _I32), _ptr(row_pos, _I32),
                                     _stream(stream)), "lmoe_route_noalloc")


def lmoe_pool(dims, x, pooler_w, x_lat, ws=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().lmoe_pool(ctypes.byref(dims), _ptr(x, _BF16), _ptr(pooler_w, _BF16), _ptr(x_lat, _BF16),
                            _ptr(ws), nbytes, _stream(stream)), "lmoe_pool")


def lmoe_experts_mxfp4(dims, x_lat, expert_offsets, sorted_rows, w13_q, w13_s, w2_q, w2_s, y, ws, stream=None):
    _check(load().lmoe_experts_mxfp4(ctypes.byref(dims), _ptr(x_lat, _BF16), _ptr(expert_offsets, _I32),
                                     _ptr(sorted_rows, _I32), _ptr(w13_q, _U8), _ptr(w13_s, _U8), _ptr(w2_q, _U8),
                                     _ptr(w2_s, _U8), _ptr(y, _F32), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "lmoe_experts_mxfp4")


def lmoe_experts_nvfp4(dims, x_lat, expert_offsets, sorted_rows, w13_q, w13_s, w13_gs, w2_q, w2_s, w2_gs, y, ws,
                       stream=None):
    """The experts on NVFP4 weights: E4M3 scales per 16 elements, fp32 global scales [E]."""
    _check(load().lmoe_experts_nvfp4(ctypes.byref(dims), _ptr(x_lat, _BF16), _ptr(expert_offsets, _I32),
                                     _ptr(sorted_rows, _I32), _ptr(w13_q, _U8), _ptr(w13_s, _U8),
                                     _ptr(w13_gs, _F32), _ptr(w2_q, _U8), _ptr(w2_s, _U8), _ptr(w2_gs, _F32),
                                     _ptr(y, _F32), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "lmoe_experts_nvfp4")


def nvfp4_of(w: dict) -> LmoeNvfp4Scales:
    """LmoeNvfp4Scales from device tensors {"w13_gs", "w2_gs"} (fp32 [E])."""
    return LmoeNvfp4Scales(_ptr(w["w13_gs"], _F32), _ptr(w["w2_gs"], _F32))


def lmoe_forward_nvfp4(dims, weights: LmoeWeights, nv: LmoeNvfp4Scales, x, out, ws, stream=None):
    """The layer with NVFP4 experts (weights.w13_s / w2_s hold the E4M3 scales)."""
    _check(load().lmoe_forward_nvfp4(ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(nv), _ptr(x, _BF16),
                                     _ptr(out, _BF16), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "lmoe_forward_nvfp4")


def lmoe_norm_combine_unpool(dims, y, topk_idx, topk_w, norm_g, unpooler_w, out, ws, stream=None):
    _check(load().lmoe_norm_combine_unpool(ctypes.byref(dims), _ptr(y, _F32), _ptr(topk_idx, _I32),
                                           _ptr(topk_w, _F32), _ptr(norm_g, _BF16), _ptr(unpooler_w, _BF16),
                                           _ptr(out, _BF16), _ptr(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)), "lmoe_norm_combine_unpool")


def lmoe_forward(dims, weights: LmoeWeights, x, out, ws, stream=None):
    _check(load().lmoe_forward(ctypes.byref(dims), ctypes.byref(weights), _ptr(x, _BF16), _ptr(out, _BF16),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "lmoe_forward")


def _host_ptr(t):
    """A pinned CPU tensor's address (the library checks that it is page-locked)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if t.is_cuda or not t.is_contiguous() or t.dtype not in _BF16:
        raise ValueError("expected a contiguous bf16 CPU tensor in pinned memory")
    return ctypes.c_void_p(t.data_ptr())


def lmoe_host_workspace_bytes(dims: LmoeDims) -> int:
    return int(load().lmoe_host_workspace_bytes(ctypes.byref(dims)))


def lmoe_forward_host(dims, weights: LmoeWeights, x_host, out_host, ws, stream=None):
    """The layer with x and out in pinned host memory (CPU tensors from
    pin_memory()); ws from lmoe_host_workspace_bytes."""
    _check(load().lmoe_forward_host(ctypes.byref(dims), ctypes.byref(weights), _host_ptr(x_host),
                                    _host_ptr(out_host), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "lmoe_forward_host")


def lmoe_forward_routed(dims, weights: LmoeWeights, x, topk_idx, topk_w, out, ws, stream=None):
    """The layer with caller-supplied routing: topk_idx int32 [T][k], topk_w fp32 [T][k]."""
    _check(load().lmoe_forward_routed(ctypes.byref(dims), ctypes.byref(weights), _ptr(x, _BF16),
                                      _ptr(topk_idx, (torch.int32,)), _ptr(topk_w, (torch.float32,)),
                                      _ptr(out, _BF16), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "lmoe_forward_routed")


def norms_of(nw: dict, eps: float) -> LmoeBlockNorms:
    """LmoeBlockNorms from device tensors {"pre_g", "post_g"} (bf16 [H]) and the norms' epsilon."""
    return LmoeBlockNorms(_ptr(nw["pre_g"], _BF16), _ptr(nw["post_g"], _BF16), float(eps))


def lmoe_block_workspace_bytes(dims: LmoeDims) -> int:
    return int(load().lmoe_block_workspace_bytes(ctypes.byref(dims)))


def lmoe_block_forward(dims, weights: LmoeWeights, norms: LmoeBlockNorms, x, y, ws, stream=None):
    """The sandwich block y = x + post_norm(layer(pre_norm(x))); y may be x."""
    _check(load().lmoe_block_forward(ctypes.byref(dims), ctypes.byref(weights), ctypes.byref(norms),
                                     _ptr(x, _BF16), _ptr(y, _BF16), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "lmoe_block_forward")


def lmoe_status_check(ws, stream=None) -> int:
    return int(load().lmoe_status_check(_ptr(ws), _stream(stream)))


def lmoe_last_launch_count() -> int:
    return int(load().lmoe_last_launch_count())


def lmoe_last_launch_name(i: int) -> str | None:
    n = load().lmoe_last_launch_name(int(i))
    return None if n is None else n.decode()


LMOE_OPT_DENSE_MIN_TOKENS = 1
LMOE_OPT_EXPERT_TC_MIN_TOKENS = 2
LMOE_OPT_FUSED_MAX_TOKENS = 3
LMOE_OPT_DOWN_Z_MAX_TOKENS = 4


def lmoe_set_option(key: int, value: int) -> int:
    """Set a regime switch (LMOE_OPT_*); returns the previous value."""
    rc = int(load().lmoe_set_option(int(key), int(value)))
    if rc < 0:
        raise LmoeError(rc, "lmoe_set_option")
    return rc


_event_array = None


def lmoe_profile_events(events):
    """Bracket launch i of the following calls with events[2i] (before) and
    events[2i + 1] (after), both on that launch's stream (None to stop).
    `events` are torch.cuda.Event(enable_timing=True) objects."""
    global _event_array
    if not events:
        _event_array = None
        _check(load().lmoe_profile_events(None, 0), "lmoe_profile_events")
        return
    for e in events:
        e.record()  # make sure the underlying CUDA event exists
    torch.cuda.synchronize()
    _event_array = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().lmoe_profile_events(_event_array, len(events)), "lmoe_profile_events")


def lmoe_selftest_timeout(ws, limit_us=10000, stream=None):
    """Enqueue a wait that nothing completes, bounded by limit_us; the status word of
    ws then reads LMOE_ETIMEOUT (lmoe_status_check)."""
    _check(load().lmoe_selftest_timeout(_ptr(ws), ws.numel() * ws.element_size(), int(limit_us), _stream(stream)),
           "lmoe_selftest_timeout")


def lmoe_selftest_e2m1(out):
    _check(load().lmoe_selftest_e2m1(_ptr(out, _F32)), "lmoe_selftest_e2m1")


def lmoe_selftest_dequant_bf16(codes, scales, out):
    """codes: uint8 [nblocks*16], scales: uint8 [nblocks], out: bf16 [nblocks*32] (device tensors)."""
    n = scales.numel()
    _check(load().lmoe_selftest_dequant_bf16(_ptr(codes), _ptr(scales), n, _ptr(out)), "lmoe_selftest_dequant_bf16")
