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

``rmsnorm``, ``rmsnorm_bwd`` and ``layer_attn`` compose these into the attention
half of a decoder layer (§The model: RMSNorm, fused QKV matmul, RoPE, attention,
output projection into the residual stream), forward and backward in f64, for the
whole-layer check of the GPU attention.
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


# ----------------------------------------------------------------------------
# The attention half of one decoder layer ("A transformer in PTX", §The model):
# RMSNorm of the residual stream, one fused matmul for q, k and v, RoPE on q and
# k, causal grouped-query attention, and the output projection added straight
# into the residual stream. Used by the whole-layer check of the GPU attention
# (the matmuls and the norm on the GPU side come from torch there). The page
# gives no epsilon for RMSNorm; 1e-5 is used, and the gain multiplies after the
# normalisation.
# ----------------------------------------------------------------------------

def rmsnorm(x, g, eps: float = 1e-5):
    """y = x / sqrt(mean(x^2 over the last axis) + eps) * g, and the per-row 1/sqrt(...)."""
    x, g = _as_f64(x), _as_f64(g)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    return x * r[..., None] * g, r


def rmsnorm_bwd(x, g, r, dy):
    """Gradients of rmsnorm with respect to x and g, given dL/dy and the forward's r:
    dx_j = g_j r dy_j - x_j r^3 / C * sum_i dy_i g_i x_i,  dg = sum over rows of dy * x * r."""
    x, g, dy = _as_f64(x), _as_f64(g), _as_f64(dy)
    C = x.shape[-1]
    dot = np.sum(dy * g * x, axis=-1)
    dx = g * r[..., None] * dy - x * (r ** 3 * dot / C)[..., None]
    dg = np.sum((dy * x * r[..., None]).reshape(-1, C), axis=0)
    return dx, dg


def layer_attn(x, g, w_qkv, w_o, Hq: int, Hkv: int, d: int, dx2, base: float = 10000.0, eps: float = 1e-5):
    """Forward and backward of the attention half of a layer, in f64.

    x [B,T,C] residual stream, g [C] norm gain, w_qkv [(Hq+2*Hkv)*d, C] (rows: q heads,
    then k heads, then v heads), w_o [C, Hq*d], dx2 [B,T,C] the upstream gradient of the
    output x2 = x + attention(rope(q), rope(k), v) w_o^T. The loss is sum(x2 * dx2).
    Returns x2 and the gradients dx, dg, dw_qkv, dw_o, plus the intermediates q, k, v
    (unrotated) and o."""
    x, g, w_qkv, w_o, dx2 = (_as_f64(a) for a in (x, g, w_qkv, w_o, dx2))
    B, T, C = x.shape
    H3 = Hq + 2 * Hkv
    xn, r = rmsnorm(x, g, eps)
    qkv = (xn.reshape(-1, C) @ w_qkv.T).reshape(B, T, H3, d)
    q, k, v = qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:]
    qr, kr = rope(q, base), rope(k, base)
    # the attention output's upstream gradient is known before the attention runs
    do = (dx2.reshape(-1, C) @ w_o).reshape(B, T, Hq, d)
    att = bwd(np.ascontiguousarray(qr), np.ascontiguousarray(kr), np.ascontiguousarray(v), do, causal=True)
    y = att["o"].reshape(B * T, Hq * d)
    x2 = x + (y @ w_o.T).reshape(B, T, C)
    dw_o = dx2.reshape(-1, C).T @ y
    dq = rope(att["dq"], base, inverse=True)
    dk = rope(att["dk"], base, inverse=True)
    dqkv = np.concatenate([dq, dk, att["dv"]], axis=2).reshape(B * T, H3 * d)
    dw_qkv = dqkv.T @ xn.reshape(-1, C)
    dxn = (dqkv @ w_qkv).reshape(B, T, C)
    dx_norm, dg = rmsnorm_bwd(x, g, r, dxn)
    return dict(x2=x2, dx=dx2 + dx_norm, dg=dg, dw_qkv=dw_qkv, dw_o=dw_o, q=q, k=k, v=v, o=att["o"])


def layer_attn_loss(x, g, w_qkv, w_o, Hq: int, Hkv: int, d: int, dx2, base: float = 10000.0, eps: float = 1e-5):
    """The scalar sum(x2 * dx2) of layer_attn's forward alone (for finite differences)."""
    x, g, w_qkv, w_o, dx2 = (_as_f64(a) for a in (x, g, w_qkv, w_o, dx2))
    B, T, C = x.shape
    H3 = Hq + 2 * Hkv
    xn, _ = rmsnorm(x, g, eps)
    qkv = (xn.reshape(-1, C) @ w_qkv.T).reshape(B, T, H3, d)
    q, k, v = qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:]
    o, _ = fwd(np.ascontiguousarray(rope(q, base)), np.ascontiguousarray(rope(k, base)), np.ascontiguousarray(v),
               causal=True)
    x2 = x + (o.reshape(B * T, Hq * d) @ w_o.T).reshape(B, T, C)
    return float(np.sum(x2 * dx2))
