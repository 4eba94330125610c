"""The oracle: a plain fp64 CPU restatement of the routed MoE layer on MXFP4 experts.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path (the
``mxfp4_routed_expert_06_b300`` package and its CUDA library) never calls it and
shares no code with it.

The arithmetic lives in ``k3oracle.c`` (plain C99, scalar, fp64; every function
cites the passage of the pages it follows).  This module only builds the library
and marshals numpy arrays.

Parity pins (tests that tie the oracle to something other than itself) are in
``tests/test_oracle_pins.py``.  Every oracle function is pinned, with two exceptions:
the end-to-end y values of full-size layers, which the pages never print (they are
pinned through the per-step pins and the second formulation of the FFN), and the
SiTU-GLU gate (``situ``, act = 1): parity unpinned, because the pages give only its
ingredients (tanh, sigmoid) and its bound (beta1 * beta2 = 100), not its formula; the
pins check the bound and the properties of the reading written in k3oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libk3oracle.so")
_SRC = os.path.join(_HERE, "k3oracle.c")


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SRC) > os.path.getmtime(_SO):
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Werror",
                               _SRC, "-o", _SO, "-lm"])
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, vp, d = ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.k3o_e2m1.argtypes, lib.k3o_e2m1.restype = [i32], d
        lib.k3o_e8m0.argtypes, lib.k3o_e8m0.restype = [i32], d
        lib.k3o_bf16.argtypes, lib.k3o_bf16.restype = [ctypes.c_uint16], d
        lib.k3o_mx_elem.argtypes, lib.k3o_mx_elem.restype = [vp, vp, i32, i32, i32], d
        lib.k3o_decode_matrix.argtypes, lib.k3o_decode_matrix.restype = [vp, vp, i32, i32, vp], None
        lib.k3o_expert_nib_bytes.argtypes, lib.k3o_expert_nib_bytes.restype = [i32, i32], ctypes.c_longlong
        lib.k3o_expert_scale_bytes.argtypes, lib.k3o_expert_scale_bytes.restype = [i32, i32], ctypes.c_longlong
        lib.k3o_router.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.k3o_router.restype = None
        lib.k3o_bucket.argtypes, lib.k3o_bucket.restype = [i32, i32, i32, vp, vp, vp, vp], None
        lib.k3o_expert_ffn.argtypes, lib.k3o_expert_ffn.restype = [i32, i32, vp, vp, vp, vp, vp, vp, i32], None
        lib.k3o_moe.argtypes, lib.k3o_moe.restype = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32], None
        lib.k3o_situ.argtypes, lib.k3o_situ.restype = [d], d
        lib.k3o_bf16_rne.argtypes, lib.k3o_bf16_rne.restype = [ctypes.c_float], ctypes.c_uint16
        lib.k3o_residual_rmsnorm.argtypes = [i32, i32, vp, vp, d, vp, vp]
        lib.k3o_residual_rmsnorm.restype = None
        lib.k3o_max_threads.argtypes, lib.k3o_max_threads.restype = [], i32
        lib.k3o_set_threads.argtypes, lib.k3o_set_threads.restype = [i32], None
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def e2m1(code: int) -> float:
    return _L().k3o_e2m1(code)


def e8m0(s: int) -> float:
    return _L().k3o_e8m0(s)


def bf16(bits: int) -> float:
    return _L().k3o_bf16(bits)


def expert_bytes(d: int, f: int) -> tuple[int, int]:
    return int(_L().k3o_expert_nib_bytes(d, f)), int(_L().k3o_expert_scale_bytes(d, f))


def mx_elem(nib, scl, cols: int, r: int, c: int) -> float:
    nib, scl = _c(nib, np.uint8), _c(scl, np.uint8)
    return _L().k3o_mx_elem(_p(nib), _p(scl), cols, r, c)


def decode_matrix(nib, scl, rows: int, cols: int) -> np.ndarray:
    nib, scl = _c(nib, np.uint8), _c(scl, np.uint8)
    assert nib.size == rows * cols // 2 and scl.size == rows * cols // 32
    out = np.empty((rows, cols), np.float64)
    _L().k3o_decode_matrix(_p(nib), _p(scl), rows, cols, _p(out))
    return out


def router(x_bits, Wr, bias, k: int):
    """-> (idx int32[T,k], w float64[T,k], logits float64[T,E], keys float64[T,E])."""
    x_bits, Wr = _c(x_bits, np.uint16), _c(Wr, np.float32)
    T, d = x_bits.shape
    E = Wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    keys = np.empty((T, E), np.float64)
    _L().k3o_router(T, d, E, k, _p(x_bits), _p(Wr), _p(b), _p(idx), _p(w), _p(logits), _p(keys))
    return idx, w, logits, keys


def topk_gap(keys: np.ndarray, k: int) -> np.ndarray:
    """Per token: k-th largest key minus (k+1)-th largest key (inf when k == E)."""
    s = -np.sort(-keys, axis=1)
    if k >= keys.shape[1]:
        return np.full(keys.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def bucket(idx, E: int):
    """-> (counts int32[E], offsets int32[E+1], perm int32[T*k])."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    _L().k3o_bucket(T, k, E, _p(idx), _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


ACT_SWIGLU, ACT_SITU_GLU = 0, 1


def situ(z: float) -> float:
    """The SiTU-GLU gate as this oracle reads it (parity unpinned: see k3oracle.c)."""
    return _L().k3o_situ(z)


def expert_ffn(d: int, f: int, nib, scl, x, act: int = ACT_SWIGLU):
    """One expert on one token (x as float64[d]) -> (h[f], o[d], a[d])."""
    nib, scl, x = _c(nib, np.uint8), _c(scl, np.uint8), _c(x, np.float64)
    h = np.empty(f, np.float64)
    o = np.empty(d, np.float64)
    a = np.empty(d, np.float64)
    _L().k3o_expert_ffn(d, f, _p(nib), _p(scl), _p(x), _p(h), _p(o), _p(a), act)
    return h, o, a


def moe(x_bits, w, pick_nib: list, pick_scl: list, f: int, act: int = ACT_SWIGLU):
    """Combine of the T*k picks.  pick_nib[p]/pick_scl[p]: canonical block of the
    expert of pick p = t*k + slot.  -> (y float64[T,d], sumabs float64[T,d])."""
    x_bits = _c(x_bits, np.uint16)
    w = _c(w, np.float64)
    T, d = x_bits.shape
    k = w.shape[1]
    assert len(pick_nib) == T * k and len(pick_scl) == T * k
    keep = [_c(a, np.uint8) for a in pick_nib] + [_c(a, np.uint8) for a in pick_scl]
    nptr = (ctypes.c_void_p * (T * k))(*[a.ctypes.data for a in keep[:T * k]])
    sptr = (ctypes.c_void_p * (T * k))(*[a.ctypes.data for a in keep[T * k:]])
    y = np.empty((T, d), np.float64)
    sumabs = np.empty((T, d), np.float64)
    _L().k3o_moe(T, d, f, k, _p(x_bits), _p(w), ctypes.addressof(nptr), ctypes.addressof(sptr), _p(y), _p(sumabs),
                 act)
    del keep
    return y, sumabs


def layer(x_bits, Wr, bias, k: int, f: int, nib_all, scl_all, act: int = ACT_SWIGLU):
    """The whole layer for configs whose experts fit in host memory.
    nib_all/scl_all: canonical blocks of all E experts, [E, ...]."""
    idx, w, logits, keys = router(x_bits, Wr, bias, k)
    counts, offsets, perm = bucket(idx, Wr.shape[0])
    flat = idx.reshape(-1)
    y, sumabs = moe(x_bits, w, [nib_all[e] for e in flat], [scl_all[e] for e in flat], f, act)
    return dict(idx=idx, w=w, logits=logits, keys=keys, counts=counts, offsets=offsets, perm=perm, y=y,
                sumabs=sumabs)


def bf16_rne(v: float) -> int:
    """float32 value -> bf16 bit pattern, round to nearest, ties to even."""
    return int(_L().k3o_bf16_rne(v))


def residual_rmsnorm(y, x_bits, eps: float):
    """Glue between stacked layers: -> (x_next uint16[T,d], x_norm uint16[T,d]) as bf16 bits."""
    y, x_bits = _c(y, np.float32), _c(x_bits, np.uint16)
    T, dd = x_bits.shape
    assert y.shape == (T, dd)
    x_next = np.empty((T, dd), np.uint16)
    x_norm = np.empty((T, dd), np.uint16)
    _L().k3o_residual_rmsnorm(T, dd, _p(y), _p(x_bits), eps, _p(x_next), _p(x_norm))
    return x_next, x_norm


def max_threads() -> int:
    return _L().k3o_max_threads()


def set_threads(n: int) -> None:
    _L().k3o_set_threads(n)
