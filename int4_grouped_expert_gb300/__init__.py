"""Python binding of libstrata.so, the GB300 routed int4-g128 MoE layer (C ABI: include/strata.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Functions carry the C names and take raw device pointers (ints) or
torch tensors (their data_ptr() is passed). The library must be built first
(`python -m int4_grouped_expert_gb300.build` or `__graft_entry__.build()`);
loading fails loudly when it is missing — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libstrata.so")

STRATA_OK = 0
STATUS_NAMES = ["STRATA_OK", "STRATA_ERR_INVALID_ARG", "STRATA_ERR_SHAPE", "STRATA_ERR_UNSUPPORTED",
                "STRATA_ERR_WORKSPACE", "STRATA_ERR_CUDA", "STRATA_ERR_DEVICE_STATUS",
                "STRATA_ERR_TIMEOUT"]
STRATA_RENORM = 0x1
STRATA_ADD_RESIDUAL = 0x2
STRATA_ROUTER_FP16 = 0x4
STRATA_FORCE_WARP_PATH = 0x100
STRATA_FORCE_TC_PATH = 0x200
STRATA_WS_REUSE = 0x8
STRATA_DEV_NONFINITE = 0x1
STRATA_DEV_BAD_ID = 0x2
STRATA_DEV_TIMEOUT = 0x4
STRATA_DEV_BAD_TOKENS = 0x8
STRATA_ERR_DEVICE_STATUS = 6
STRATA_ERR_TIMEOUT = 7
GROUP_WORKSPACE_BYTES = 256
GROUP = 128


class StrataError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name}")


class strata_moe_layer(ctypes.Structure):
    """Mirror of the C struct strata_moe_layer."""
    _fields_ = [
        ("H", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
        ("has_shared", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("w_router", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("gate_codes", ctypes.c_void_p), ("gate_scales", ctypes.c_void_p),
        ("up_codes", ctypes.c_void_p), ("up_scales", ctypes.c_void_p),
        ("down_codes", ctypes.c_void_p), ("down_scales", ctypes.c_void_p),
        ("group_size", ctypes.c_int32), ("bits", ctypes.c_int32),
    ]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U32 = ctypes.c_uint32
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "strata_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "strata_version": (ctypes.c_int, []),
    "strata_quantize_groups": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P, _P]),
    "strata_quantize_groups_bits": (ctypes.c_int, [_P, _I64, _I64, _I32, _I32, _P, _P, _P, _P]),
    "strata_route_workspace_size": (_SZ, [_I64, _I32, _I32]),
    "strata_route_topk": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _I32, _U32,
                                         _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "strata_route_topk_noalloc": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _I32, _U32,
                                                 _P, _P, _P, _P, _P, _P, _P]),
    "strata_moe_workspace_size": (_SZ, [ctypes.POINTER(strata_moe_layer), _I64]),
    "strata_moe_forward": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _I64, _P, _P, _SZ, _P]),
    "strata_moe_forward_padded": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _P, _I64,
                                                 _P, _P, _SZ, _P]),
    "strata_group_rows": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "strata_selftest_bounded_waits": (ctypes.c_int, [_P, _I64, _P]),
    "strata_moe_forward_ex": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _I64, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "strata_moe_forward_stats": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _I64, _P, _P,
                                                 _P, _SZ, _P]),
    "strata_moe_forward_profiled": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _I64, _P, _P,
                                                   _SZ, _P, ctypes.POINTER(_P), _I32]),
    "strata_moe_stack_workspace_size": (_SZ, [ctypes.POINTER(strata_moe_layer), _I32, _I64]),
    "strata_moe_stack_forward": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _I32, _P, _I64,
                                                _P, _P, _SZ, _P]),
    "strata_moe_host_staging_size": (_SZ, [ctypes.POINTER(strata_moe_layer), _I64]),
    "strata_moe_forward_host": (ctypes.c_int, [ctypes.POINTER(strata_moe_layer), _P, _I64, _P, _P,
                                               _SZ, _P]),
    "strata_workspace_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(_U32)]),
    "strata_read_status": (ctypes.c_int, [_P, _P, ctypes.POINTER(_U32)]),
}


def lib() -> ctypes.CDLL:
    """Load libstrata.so (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m int4_grouped_expert_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def ptr(t) -> int | None:
    """Device pointer of a torch tensor (or pass through an int / None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def stream_handle(stream) -> int | None:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:  # pragma: no cover
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(status: int, where: str) -> None:
    if status != STRATA_OK:
        raise StrataError(status, where)


# ----------------------------------------------------------------------------- the C calls

def strata_status_string(status: int) -> str:
    return lib().strata_status_string(status).decode()


def strata_version() -> int:
    return lib().strata_version()


def strata_quantize_groups(w, n, k, codes, scales, dev_status=None, group_size=GROUP, stream=None):
    return lib().strata_quantize_groups(ptr(w), n, k, group_size, ptr(codes), ptr(scales),
                                        ptr(dev_status), stream_handle(stream))


def strata_quantize_groups_bits(w, n, k, codes, scales, dev_status=None, group_size=GROUP, bits=4,
                                stream=None):
    return lib().strata_quantize_groups_bits(ptr(w), n, k, group_size, bits, ptr(codes),
                                             ptr(scales), ptr(dev_status), stream_handle(stream))


def strata_route_workspace_size(T, E, k) -> int:
    return lib().strata_route_workspace_size(T, E, k)


def strata_route_topk(x, w_router, bias, T, H, E, k, flags, ids, gates, counts=None, offsets=None,
                      perm=None, inv=None, workspace=None, ws_bytes=0, stream=None):
    return lib().strata_route_topk(ptr(x), ptr(w_router), ptr(bias), T, H, E, k, flags, ptr(ids),
                                   ptr(gates), ptr(counts), ptr(offsets), ptr(perm), ptr(inv),
                                   ptr(workspace), ws_bytes, stream_handle(stream))


def strata_route_topk_noalloc(x, w_router, bias, T, H, E, k, flags, ids, gates, counts=None,
                              offsets=None, perm=None, inv=None, stream=None):
    """strata_route_topk with the library's own fixed scratch (no workspace, no allocation)."""
    return lib().strata_route_topk_noalloc(ptr(x), ptr(w_router), ptr(bias), T, H, E, k, flags,
                                           ptr(ids), ptr(gates), ptr(counts), ptr(offsets),
                                           ptr(perm), ptr(inv), stream_handle(stream))


NOALLOC_SCRATCH_BYTES = 8 << 20


def strata_moe_workspace_size(layer: strata_moe_layer, T_max: int) -> int:
    return lib().strata_moe_workspace_size(ctypes.byref(layer), T_max)


def strata_moe_forward(layer, x, T, out, workspace, ws_bytes, stream=None):
    return lib().strata_moe_forward(ctypes.byref(layer), ptr(x), T, ptr(out), ptr(workspace),
                                    ws_bytes, stream_handle(stream))


def strata_moe_forward_padded(layer, x, n_tokens, T_max, out, workspace, ws_bytes, stream=None):
    """n_tokens: a device int32 (tensor or pointer) holding the live token count."""
    return lib().strata_moe_forward_padded(ctypes.byref(layer), ptr(x), ptr(n_tokens), T_max, ptr(out),
                                           ptr(workspace), ws_bytes, stream_handle(stream))


def strata_group_rows(ids, T, k, E, counts, offsets, perm, inv, workspace, ws_bytes, stream=None):
    return lib().strata_group_rows(ptr(ids), T, k, E, ptr(counts), ptr(offsets), ptr(perm), ptr(inv),
                                   ptr(workspace), ws_bytes, stream_handle(stream))


def strata_selftest_bounded_waits(dev_words, limit_cycles, stream=None):
    return lib().strata_selftest_bounded_waits(ptr(dev_words), limit_cycles, stream_handle(stream))


def strata_moe_forward_stats(layer, x, T, out, expert_rows, workspace, ws_bytes, stream=None):
    return lib().strata_moe_forward_stats(ctypes.byref(layer), ptr(x), T, ptr(out), ptr(expert_rows),
                                          ptr(workspace), ws_bytes, stream_handle(stream))


def strata_moe_forward_ex(layer, x, T, out, ids=None, gates=None, counts=None, offsets=None,
                          perm=None, inv=None, workspace=None, ws_bytes=0, stream=None):
    return lib().strata_moe_forward_ex(ctypes.byref(layer), ptr(x), T, ptr(out), ptr(ids), ptr(gates),
                                       ptr(counts), ptr(offsets), ptr(perm), ptr(inv),
                                       ptr(workspace), ws_bytes, stream_handle(stream))


def strata_moe_forward_profiled(layer, x, T, out, workspace, ws_bytes, events, stream=None):
    """events: 6 torch.cuda.Event objects (or raw cudaEvent_t ints / None)."""
    handles = (_P * len(events))(*[None if e is None else (e if isinstance(e, int) else e.cuda_event)
                                   for e in events])
    return lib().strata_moe_forward_profiled(ctypes.byref(layer), ptr(x), T, ptr(out),
                                             ptr(workspace), ws_bytes, stream_handle(stream),
                                             handles, len(events))


def layer_array(structs):
    """A C array of strata_moe_layer from a list of descriptors."""
    arr = (strata_moe_layer * len(structs))(*structs)
    return arr


def strata_moe_stack_workspace_size(layers, T_max) -> int:
    arr = layers if not isinstance(layers, list) else layer_array(layers)
    return lib().strata_moe_stack_workspace_size(arr, len(arr), T_max)


def strata_moe_stack_forward(layers, x, T, out, workspace, ws_bytes, stream=None):
    arr = layers if not isinstance(layers, list) else layer_array(layers)
    return lib().strata_moe_stack_forward(arr, len(arr), ptr(x), T, ptr(out), ptr(workspace),
                                          ws_bytes, stream_handle(stream))


def strata_moe_host_staging_size(layer, T_max) -> int:
    return lib().strata_moe_host_staging_size(ctypes.byref(layer), T_max)


def strata_moe_forward_host(layer, x_host, T, out_host, workspace, ws_bytes, stream=None):
    return lib().strata_moe_forward_host(ctypes.byref(layer), ptr(x_host), T, ptr(out_host),
                                         ptr(workspace), ws_bytes, stream_handle(stream))


def strata_workspace_status(workspace, stream=None):
    v = _U32(0)
    st = lib().strata_workspace_status(ptr(workspace), stream_handle(stream), ctypes.byref(v))
    return st, v.value


def strata_read_status(dev_status, stream=None):
    v = _U32(0)
    st = lib().strata_read_status(ptr(dev_status), stream_handle(stream), ctypes.byref(v))
    return st, v.value


from .layer import MoELayer  # noqa: E402,F401
