"""CPU oracle for causal grouped-query attention (forward and backward, f64).

TEST INFRASTRUCTURE. This package checks the CUDA library; it is not part of
it. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It shares no code with ``causal_gqa_flash_gb300``.

What it computes is the plain definition of attention that the flash kernels
of "A transformer in PTX" (§Flash attention, §The same bits every time) reach
by tiles; the formulas are listed at the top of ``oracle.c``. Arrays are numpy
float64, C-contiguous, with q/o/dO/dq in [B,T,Hq,d], k/v/dk/dv in [B,T,Hkv,d]
and lse/D in [B,Hq,T] (natural-log LSE).

``rope`` is the rotary position embedding that the trainer applies to the
queries and keys before attention ("A transformer in PTX", §The model); the
page names it and gives no formula, so it is the textbook rotation (pairs of
adjacent features, frequencies base^(-2i/d), angle = token index), written
out below in numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None

_D = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (portable flags, OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i = ctypes.c_int
        lib.oracle_fwd.argtypes = [_D, _D, _D, _D, _D, i, i, i, i, i, i, ctypes.c_double, i]
        lib.oracle_bwd.argtypes = [_D] * 10 + [i, i, i, i, i, i, ctypes.c_double, i]
        lib.oracle_probs.argtypes = [_D, _D, i, i, i, i, i, i, ctypes.c_double, i, i, _D, _D, i]
        lib.oracle_max_threads.argtypes = []
        for f in (lib.oracle_fwd, lib.oracle_bwd, lib.oracle_probs, lib.oracle_max_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_D)


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _shape(q, k):
    B, T, Hq, d = q.shape
    Bk, Tk, Hkv, dk = k.shape
    if (B, T, d) != (Bk, Tk, dk):
        raise ValueError(f"q {q.shape} and k {k.shape} disagree")
    return B, T, Hq, Hkv, d


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def fwd(q, k, v, causal: bool = True, scale: float | None = None, threads: int = 0):
    """Return (O [B,T,Hq,d], LSE [B,Hq,T]) in float64."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, T, Hq, Hkv, d = _shape(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, T), dtype=np.float64)
    rc = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, Hq, Hkv, d,
                            int(bool(causal)), float(scale), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_fwd failed ({rc})")
    return o, lse


def bwd(q, k, v, dout, causal: bool = True, scale: float | None = None, threads: int = 0):
    """Return dict with o, lse, D, dq, dk, dv (float64) for the loss sum(O * dO)."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, T, Hq, Hkv, d = _shape(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, T), dtype=np.float64)
    D = np.empty((B, Hq, T), dtype=np.float64)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse), _ptr(D), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, T, Hq, Hkv, d, int(bool(causal)), float(scale),
                            int(threads))
    if rc != 0:
        raise ValueError(f"oracle_bwd failed ({rc})")
    return dict(o=o, lse=lse, D=D, dq=dq, dk=dk, dv=dv)


def probs(q, k, b: int, h: int, causal: bool = True, scale: float | None = None, threads: int = 0):
    """Return (P [T,T], LSE [T]) of query head h in batch b."""
    q, k = _as_f64(q), _as_f64(k)
    B, T, Hq, Hkv, d = _shape(q, k)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    P = np.empty((T, T), dtype=np.float64)
    lse = np.empty((T,), dtype=np.float64)
    rc = _load().oracle_probs(_ptr(q), _ptr(k), B, T, Hq, Hkv, d, int(bool(causal)), float(scale), int(b),
                              int(h), _ptr(P), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_probs failed ({rc})")
    return P, lse


def rope_angles(T: int, d: int, base: float = 10000.0) -> np.ndarray:
    """Angles [T, d/2] of the rotary embedding: angle[t, i] = t * base**(-2i/d)."""
    if d % 2:
        raise ValueError("d must be even")
    theta = base ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)
    return np.arange(T, dtype=np.float64)[:, None] * theta[None, :]


def rope(x, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotary embedding of x [B, T, H, d] in float64.

    Feature pair (2i, 2i+1) of token t is rotated by angle[t, i] (``rope_angles``):
        y[2i]   = x[2i] cos - x[2i+1] sin
        y[2i+1] = x[2i] sin + x[2i+1] cos
    ``inverse`` rotates by minus the angle (the transpose), which is also the
    gradient of the rotation: dx = rope(dy, inverse=True).
    """
    x = _as_f64(x)
    B, T, H, d = x.shape
    ang = rope_angles(T, d, base)
    c = np.cos(ang)[None, :, None, :]
    s = np.sin(ang)[None, :, None, :]
    if inverse:
        s = -s
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y
