"""Routed mixture-of-experts layer on MXFP4 experts for B300 (sm_103a).

A thin ctypes binding of ``libk3moe.so``; every function has the name of the C entry
point it marshals (declared and documented in ``include/k3moe.h``).  Arguments may be
torch tensors (their ``data_ptr()`` is passed), numpy arrays (host pointers), raw
integer pointers, or ``None`` for NULL.  Streams may be ``torch.cuda.Stream``, an
integer ``cudaStream_t`` or ``None`` (the current torch stream when torch is loaded,
else the legacy default stream).

No computation happens in Python: every step of the layer runs in the library's CUDA
kernels.  The package refuses to import when ``libk3moe.so`` has not been built
(``python mxfp4_routed_expert_06_b300/build.py``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libk3moe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "k3moe.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python mxfp4_routed_expert_06_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)


def _header_constants() -> dict:
    out = {}
    with open(HEADER) as fh:
        for m in re.finditer(r"#define\s+(K3MOE_\w+)\s+\(?(-?(?:0x[0-9A-Fa-f]+|\d+))u?\)?", fh.read()):
            out[m.group(1)] = int(m.group(2), 0)
    return out


_C = _header_constants()
globals().update(_C)
K3MOE_K_COUNT = 9
KERNEL_NAMES = ["router", "topk", "bucket", "gateup", "down", "gemm_gu", "gemm_dn", "combine", "gather"]


class k3moe_dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("f", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("T_max", ctypes.c_int)]


class k3moe_cache_stats_t(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64),
                ("h2d_bytes", ctypes.c_uint64), ("h2d_ms", ctypes.c_double), ("calls", ctypes.c_uint64),
                ("prefetched", ctypes.c_uint64)]


class k3moe_cache_sim_stats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_longlong), ("misses", ctypes.c_longlong), ("evictions", ctypes.c_longlong)]


class k3moe_pool_header(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("d", ctypes.c_int32),
                ("f", ctypes.c_int32), ("E", ctypes.c_int32), ("s_min", ctypes.c_int32), ("s_max", ctypes.c_int32),
                ("zero_scales", ctypes.c_int32), ("expert_bytes", ctypes.c_uint64), ("checksum", ctypes.c_uint64)]


class k3moe_kernel_time(ctypes.Structure):
    _fields_ = [("ms_total", ctypes.c_double), ("launches", ctypes.c_longlong)]


_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "k3moe_packed_expert_bytes": ([ctypes.POINTER(k3moe_dims)], _sz),
    "k3moe_pack_experts": ([ctypes.POINTER(k3moe_dims), _vp, _vp, _i, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)], _i),
    "k3moe_router_topk": ([_vp, _vp, _i, _vp, _vp, _vp], _i),
    "k3moe_bucket": ([_vp, _vp, _i, _vp, _vp, _vp, _vp], _i),
    "k3moe_layer_forward": ([_vp, _vp, _i, _vp, _vp], _i),
    "k3moe_layer_forward_host": ([_vp, _vp, _i, _vp, _vp], _i),
    "k3moe_graph_create": ([_vp, _vp, _i, _i, _vp, _vp, ctypes.POINTER(_vp)], _i),
    "k3moe_graph_launch": ([_vp, _vp], _i),
    "k3moe_graph_destroy": ([_vp], None),
    "k3moe_set_option": ([_vp, _i, ctypes.c_longlong], _i),
    "k3moe_sync": ([_vp], _i),
    "k3moe_profile": ([_vp, _i], _i),
    "k3moe_profile_read": ([_vp, ctypes.POINTER(k3moe_kernel_time)], _i),
    "k3moe_read_packed": ([_vp, _i, _vp], _i),
    "k3moe_debug_buffer": ([_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_sz)], _i),
    "k3moe_layer_free": ([_vp], None),
    "k3moe_cache_create": ([_sz, _sz, ctypes.POINTER(_vp)], _i),
    "k3moe_cache_stats": ([_vp, ctypes.POINTER(k3moe_cache_stats_t)], _i),
    "k3moe_cache_reset_stats": ([_vp], _i),
    "k3moe_cache_destroy": ([_vp], None),
    "k3moe_layer_set_cache": ([_vp, _vp], _i),
    "k3moe_residual_rmsnorm": ([_vp, _vp, _i, _i, ctypes.c_float, _vp, _vp, _vp], _i),
    "k3moe_cache_simulate": ([_vp, _vp, _i, _i, _i, ctypes.c_ulonglong, ctypes.POINTER(k3moe_cache_sim_stats)], _i),
    "k3moe_last_error": ([], ctypes.c_char_p),
    "k3moe_router_topk_noalloc": ([_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp], _i),
    "k3moe_cache_set_device_lru": ([_vp, _i], _i),
    "k3moe_cache_prefetch": ([_vp, _vp, _i, ctypes.POINTER(_i)], _i),
    "k3moe_pool_header_get": ([_vp, ctypes.POINTER(k3moe_pool_header)], _i),
    "k3moe_pool_header_check": ([ctypes.POINTER(k3moe_pool_header), ctypes.POINTER(k3moe_dims)], _i),
    "k3moe_layer_from_packed": ([ctypes.POINTER(k3moe_dims), ctypes.POINTER(k3moe_pool_header), _vp, _i, _vp, _vp,
                                 _vp, _vp, ctypes.POINTER(_vp)], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def exported_symbols() -> list[str]:
    return sorted(_SIGS)


class K3MoEError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"k3moe error {code}: {msg}")
        self.code = code


def k3moe_last_error() -> str:
    return _lib.k3moe_last_error().decode()


def _check(rc: int) -> None:
    if rc != 0:
        raise K3MoEError(rc, k3moe_last_error())


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _handle(h):
    return h.value if isinstance(h, ctypes.c_void_p) else h


def dims(d: int, f: int, E: int, k: int, T_max: int) -> k3moe_dims:
    return k3moe_dims(d, f, E, k, T_max)


def k3moe_packed_expert_bytes(dm: k3moe_dims) -> int:
    return _lib.k3moe_packed_expert_bytes(ctypes.byref(dm))


def k3moe_pack_experts(dm: k3moe_dims, canon_nib, canon_scale, src_on_device: int, W_r, bias=None, cache=None,
                       stream=None):
    out = ctypes.c_void_p()
    _check(_lib.k3moe_pack_experts(ctypes.byref(dm), _ptr(canon_nib), _ptr(canon_scale), int(src_on_device),
                                   _ptr(W_r), _ptr(bias), _handle(cache), _stream(stream), ctypes.byref(out)))
    return out


def k3moe_pool_header_get(layer) -> k3moe_pool_header:
    h = k3moe_pool_header()
    _check(_lib.k3moe_pool_header_get(_handle(layer), ctypes.byref(h)))
    return h


def k3moe_pool_header_check(header: k3moe_pool_header, dm: k3moe_dims) -> None:
    _check(_lib.k3moe_pool_header_check(ctypes.byref(header), ctypes.byref(dm)))


def k3moe_layer_from_packed(dm: k3moe_dims, header: k3moe_pool_header, packed, src_on_device: int, W_r, bias=None,
                            cache=None, stream=None):
    out = ctypes.c_void_p()
    _check(_lib.k3moe_layer_from_packed(ctypes.byref(dm), ctypes.byref(header), _ptr(packed), int(src_on_device),
                                        _ptr(W_r), _ptr(bias), _handle(cache), _stream(stream), ctypes.byref(out)))
    return out


def k3moe_router_topk(layer, x, T: int, idx, w, stream=None) -> None:
    _check(_lib.k3moe_router_topk(_handle(layer), _ptr(x), T, _ptr(idx), _ptr(w), _stream(stream)))


def k3moe_bucket(layer, idx, T: int, counts, offsets, perm, stream=None) -> None:
    _check(_lib.k3moe_bucket(_handle(layer), _ptr(idx), T, _ptr(counts), _ptr(offsets), _ptr(perm), _stream(stream)))


def k3moe_layer_forward(layer, x, T: int, y, stream=None) -> None:
    _check(_lib.k3moe_layer_forward(_handle(layer), _ptr(x), T, _ptr(y), _stream(stream)))


def k3moe_layer_forward_host(layer, x_host, T: int, y_host, stream=None) -> None:
    _check(_lib.k3moe_layer_forward_host(_handle(layer), _ptr(x_host), T, _ptr(y_host), _stream(stream)))


def k3moe_sync(layer) -> None:
    _check(_lib.k3moe_sync(_handle(layer)))


def k3moe_set_option(layer, option: int, value: int) -> None:
    _check(_lib.k3moe_set_option(_handle(layer), option, value))


def k3moe_profile(layer, enable: bool) -> None:
    _check(_lib.k3moe_profile(_handle(layer), int(enable)))


def k3moe_profile_read(layer) -> dict:
    arr = (k3moe_kernel_time * K3MOE_K_COUNT)()
    _check(_lib.k3moe_profile_read(_handle(layer), arr))
    return {KERNEL_NAMES[i]: (arr[i].ms_total, arr[i].launches) for i in range(K3MOE_K_COUNT)}


def k3moe_read_packed(layer, e: int, dst) -> None:
    _check(_lib.k3moe_read_packed(_handle(layer), e, _ptr(dst)))


def k3moe_debug_buffer(layer, which: int) -> tuple[int, int]:
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check(_lib.k3moe_debug_buffer(_handle(layer), which, ctypes.byref(ptr), ctypes.byref(n)))
    return ptr.value, n.value


def k3moe_layer_free(layer) -> None:
    _lib.k3moe_layer_free(_handle(layer))


def k3moe_router_topk_noalloc(x, W_r, bias, T: int, d: int, E: int, k: int, idx, w, stream=None) -> None:
    _check(_lib.k3moe_router_topk_noalloc(_ptr(x), _ptr(W_r), _ptr(bias), T, d, E, k, _ptr(idx), _ptr(w),
                                          _stream(stream)))


def k3moe_graph_create(layer, x, T: int, calls: int, y, stream=None):
    """`calls` layer calls of T tokens (x, y contiguous over the calls) run once and captured as one
    CUDA graph; returns its handle for k3moe_graph_launch."""
    out = ctypes.c_void_p()
    _check(_lib.k3moe_graph_create(_handle(layer), _ptr(x), T, calls, _ptr(y), _stream(stream), ctypes.byref(out)))
    return out


def k3moe_graph_launch(graph, stream=None) -> None:
    _check(_lib.k3moe_graph_launch(_handle(graph), _stream(stream)))


def k3moe_graph_destroy(graph) -> None:
    _lib.k3moe_graph_destroy(_handle(graph))


def k3moe_cache_create(budget_bytes: int, slot_bytes: int):
    out = ctypes.c_void_p()
    _check(_lib.k3moe_cache_create(budget_bytes, slot_bytes, ctypes.byref(out)))
    return out


def k3moe_cache_stats(cache) -> dict:
    st = k3moe_cache_stats_t()
    _check(_lib.k3moe_cache_stats(_handle(cache), ctypes.byref(st)))
    return {n: getattr(st, n) for n, _ in st._fields_}


def k3moe_cache_set_device_lru(cache, enable: int) -> None:
    _check(_lib.k3moe_cache_set_device_lru(_handle(cache), int(enable)))


def k3moe_cache_prefetch(layer, experts) -> int:
    """Makes the listed experts of a cache-mode layer resident ahead of use; returns how many were
    copied (fewer than the missing ones when the remaining slots belong to calls still in flight)."""
    import numpy as np
    ids = np.ascontiguousarray(np.asarray(experts, dtype=np.int32).reshape(-1))
    got = _i(0)
    _check(_lib.k3moe_cache_prefetch(_handle(layer), ids.ctypes.data if ids.size else None, int(ids.size),
                                     ctypes.byref(got)))
    return got.value


def k3moe_cache_reset_stats(cache) -> None:
    _check(_lib.k3moe_cache_reset_stats(_handle(cache)))


def k3moe_cache_destroy(cache) -> None:
    _lib.k3moe_cache_destroy(_handle(cache))


def k3moe_residual_rmsnorm(y, x, T: int, d: int, eps: float, x_next, x_norm, stream=None) -> None:
    _check(_lib.k3moe_residual_rmsnorm(_ptr(y), _ptr(x), T, d, eps, _ptr(x_next), _ptr(x_norm), _stream(stream)))


def k3moe_cache_simulate(calls, n_slots: int, policy: int, seed: int = 0) -> dict:
    """calls: a sequence of calls, each a sequence of int expert keys (distinct within a call), in
    the order the call looks them up.  Host only.  Returns {hits, misses, evictions}."""
    import numpy as np
    starts = np.zeros(len(calls) + 1, dtype=np.int64)
    starts[1:] = np.cumsum([len(c) for c in calls])
    keys = np.ascontiguousarray(np.concatenate([np.asarray(c, dtype=np.int64) for c in calls])
                                if len(calls) else np.zeros(0, dtype=np.int64))
    st = k3moe_cache_sim_stats()
    _check(_lib.k3moe_cache_simulate(keys.ctypes.data, starts.ctypes.data, len(calls), n_slots, policy, seed,
                                     ctypes.byref(st)))
    return {n: getattr(st, n) for n, _ in st._fields_}


def k3moe_layer_set_cache(layer, cache) -> None:
    _check(_lib.k3moe_layer_set_cache(_handle(layer), _handle(cache)))
