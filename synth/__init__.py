"""Seeded, counter-based synthetic inputs for the routed MoE layer.

This package defines the inputs that the CPU oracle, the tests and the benchmark
share.  It holds none of the layer's arithmetic: no decoding, routing or FFN.
Every value is a pure function of (seed, layer, expert/token, index); see
``k3synth.h`` for the stream definitions (splitmix64 counters).

Two shared libraries are built from this folder:
  * ``libk3synth_host.so`` (gcc): every stream, on the host;
  * ``libk3synth_dev.so`` (nvcc, sm_103a): the integer expert streams, written
    straight into device memory.  Its output is bit-identical to the host one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libk3synth_host.so")
_DEV_SO = os.path.join(_HERE, "libk3synth_dev.so")

NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build_host(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, "k3synth.c"), os.path.join(_HERE, "k3synth.h")]
    if force or _stale(_HOST_SO, srcs):
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Werror",
                               srcs[0], "-o", _HOST_SO, "-lm"])
    return _HOST_SO


def build_dev(force: bool = False) -> str:
    srcs = [os.path.join(_HERE, "k3synth_dev.cu"), os.path.join(_HERE, "k3synth.h")]
    if force or _stale(_DEV_SO, srcs):
        subprocess.check_call(["nvcc", *NVCC_ARCH, "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
                               srcs[0], "-o", _DEV_SO])
    return _DEV_SO


def build(force: bool = False) -> None:
    build_host(force)
    build_dev(force)


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        u64, i32, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
        lib.k3s_experts.argtypes = [u64, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.k3s_tokens_bf16.argtypes = [u64, i32, i32, i32, i32, vp, vp]
        lib.k3s_router_weights.argtypes = [u64, i32, i32, i32, vp]
        lib.k3s_hot_experts.argtypes = [u64, i32, i32, i32, vp]
        for f in (lib.k3s_experts, lib.k3s_tokens_bf16, lib.k3s_router_weights, lib.k3s_hot_experts):
            f.restype = None
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_dev())
        lib.k3s_dev_experts.argtypes = [ctypes.c_uint64] + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 3
        lib.k3s_dev_experts.restype = ctypes.c_int
        _dev = lib
    return _dev


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def expert_bytes(d: int, f: int) -> tuple[int, int]:
    """(nibble bytes, scale bytes) of one expert in the canonical layout."""
    return 3 * f * d // 2, 3 * f * d // 32


def experts(seed: int, layer: int, e0: int, e1: int, d: int, f: int, scale_lo: int = 121, scale_hi: int = 125):
    """Canonical MXFP4 bytes of experts [e0, e1): (nib uint8[n, 3*f*d/2], scl uint8[n, 3*f*d/32])."""
    n = e1 - e0
    nb, sb = expert_bytes(d, f)
    nib = np.empty((n, nb), np.uint8)
    scl = np.empty((n, sb), np.uint8)
    _host_lib().k3s_experts(seed, layer, e0, e1, d, f, scale_lo, scale_hi, _ptr(nib), _ptr(scl))
    return nib, scl


def experts_to_device(seed: int, layer: int, e0: int, e1: int, d: int, f: int, nib_dev: int, scl_dev: int,
                      stream: int = 0, scale_lo: int = 121, scale_hi: int = 125) -> None:
    """Write the same bytes as :func:`experts` into device buffers (raw pointers)."""
    rc = _dev_lib().k3s_dev_experts(seed, layer, e0, e1, d, f, scale_lo, scale_hi, nib_dev, scl_dev, stream)
    if rc != 0:
        raise RuntimeError(f"k3s_dev_experts failed ({rc})")


def tokens_bf16(seed: int, layer: int, t0: int, T: int, d: int, attempts=None) -> np.ndarray:
    """x[T, d] as bf16 bit patterns (uint16), tokens t0..t0+T-1, N(0,1) before rounding."""
    out = np.empty((T, d), np.uint16)
    att = None
    if attempts is not None:
        att = np.ascontiguousarray(attempts, dtype=np.int32)
        assert att.shape == (T,)
    _host_lib().k3s_tokens_bf16(seed, layer, t0, T, d, None if att is None else _ptr(att), _ptr(out))
    return out


def router_weights(seed: int, layer: int, E: int, d: int) -> np.ndarray:
    """W_r[E, d] float32, N(0, 1/d)."""
    out = np.empty((E, d), np.float32)
    _host_lib().k3s_router_weights(seed, layer, E, d, _ptr(out))
    return out


def hot_bias(seed: int, layer: int, E: int, n_hot: int, value: float = 2.0) -> np.ndarray:
    """Router selection bias[E]: `value` on a seeded subset of n_hot experts, 0 elsewhere."""
    hot = np.empty(n_hot, np.int32)
    _host_lib().k3s_hot_experts(seed, layer, E, n_hot, _ptr(hot))
    b = np.zeros(E, np.float32)
    b[hot] = value
    return b


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)
