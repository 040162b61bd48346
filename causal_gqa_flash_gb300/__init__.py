"""Causal grouped-query flash attention (forward and backward) for GB300 / sm_103a.

A thin ctypes binding over the C ABI declared in ``include/gqa_attn.h``. The
functions below only marshal arguments: torch provides device memory and the
current stream, and every step of the computation runs in the library's CUDA
kernels. There is no CPU fallback: if the compiled library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes
import os

from ._build import build, library_path

__all__ = [
    "AttnError", "build", "library_path", "load", "attn_fwd", "attn_bwd", "attn_fwd_strided", "attn_bwd_strided",
    "attn_bwd_workspace_bytes",
    "attn_bwd_preprocess", "attn_bwd_dq", "attn_bwd_dkv", "attn_bwd_dq_dkv", "attn_bwd_noalloc",
    "NOALLOC_SCRATCH_BYTES",
    "attn_sync_status", "attn_selftest_timeout", "attn_set_wait_budget_ns", "attn_set_task_order", "attn_last_error", "attn_version",
    "GqaView", "view_of", "attn_rope_table", "attn_rope", "attn_fwd_rope", "attn_bwd_rope", "attn_fwd_naive", "attn_bwd_naive",
    "attn_naive_workspace_bytes", "probe_rates", "probe_tma", "EXPORTED_SYMBOLS", "GQA_OK", "GQA_ERR_INVALID_ARG", "GQA_ERR_UNSUPPORTED_DEVICE", "GQA_ERR_LAUNCH",
    "GQA_ERR_TIMEOUT",
]

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED_DEVICE = 2
GQA_ERR_LAUNCH = 3
GQA_ERR_TIMEOUT = 4
NOALLOC_SCRATCH_BYTES = 8 << 20  # GQA_NOALLOC_SCRATCH_BYTES in include/gqa_attn.h

# Every function include/gqa_attn.h declares.
EXPORTED_SYMBOLS = (
    "attn_fwd", "attn_bwd_workspace_bytes", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_dq", "attn_bwd_dkv",
    "attn_bwd_dq_dkv", "attn_bwd_noalloc", "attn_fwd_strided", "attn_bwd_strided", "attn_rope_table_bytes",
    "attn_rope_table", "attn_rope", "attn_fwd_rope", "attn_bwd_rope", "attn_naive_workspace_bytes", "attn_fwd_naive", "attn_bwd_naive",
    "attn_last_error", "attn_sync_status", "attn_selftest_timeout",
    "attn_set_wait_budget_ns", "attn_set_task_order", "attn_version", "attn_probe_mma", "attn_probe_ex2",
    "attn_probe_tma",
)

_lib = None


class GqaView(ctypes.Structure):
    """gqa_view_t: a bf16 [B, T, H, d] tensor with packed heads and free token / batch strides (elements)."""
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_t", ctypes.c_longlong), ("stride_b", ctypes.c_longlong)]


class AttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built ({path} missing): call causal_gqa_flash_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i, sz, ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_ulonglong
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.attn_fwd.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_bwd.argtypes = [vp] * 10 + [sz, i, i, i, i, i, i, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_preprocess.argtypes = [vp, vp, vp, vp, sz, i, i, i, i, vp]
    lib.attn_bwd_preprocess.restype = i
    lib.attn_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_dq.restype = i
    lib.attn_bwd_dkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_dkv.restype = i
    lib.attn_bwd_dq_dkv.argtypes = [vp] * 8 + [sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_dq_dkv.restype = i
    lib.attn_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, i, vp]
    lib.attn_bwd_noalloc.restype = i
    gv = GqaView
    lib.attn_fwd_strided.argtypes = [gv, gv, gv, gv, vp, i, i, i, i, i, i, vp]
    lib.attn_fwd_strided.restype = i
    lib.attn_bwd_strided.argtypes = [gv, gv, gv, gv, vp, gv, gv, gv, gv, vp, sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_strided.restype = i
    lib.attn_rope_table_bytes.argtypes = [i, i]
    lib.attn_rope_table_bytes.restype = sz
    lib.attn_rope_table.argtypes = [vp, i, i, ctypes.c_double, vp]
    lib.attn_rope_table.restype = i
    lib.attn_rope.argtypes = [gv, gv, vp, i, i, i, i, i, vp]
    lib.attn_rope.restype = i
    dbl = ctypes.c_double
    lib.attn_fwd_rope.argtypes = [gv, gv, gv, gv, vp, gv, gv, dbl, i, i, i, i, i, i, vp]
    lib.attn_fwd_rope.restype = i
    lib.attn_bwd_rope.argtypes = [gv, gv, gv, gv, vp, gv, gv, gv, gv, dbl, vp, sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_rope.restype = i
    lib.attn_naive_workspace_bytes.argtypes = [i, i, i]
    lib.attn_naive_workspace_bytes.restype = sz
    lib.attn_fwd_naive.argtypes = [vp] * 6 + [sz, i, i, i, i, i, i, vp]
    lib.attn_fwd_naive.restype = i
    lib.attn_bwd_naive.argtypes = [vp] * 10 + [sz, i, i, i, i, i, i, vp]
    lib.attn_bwd_naive.restype = i
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_sync_status.argtypes = [vp]
    lib.attn_sync_status.restype = i
    lib.attn_selftest_timeout.argtypes = [ull, vp]
    lib.attn_selftest_timeout.restype = i
    lib.attn_set_wait_budget_ns.argtypes = [ull]
    lib.attn_set_wait_budget_ns.restype = None
    lib.attn_set_task_order.argtypes = [i]
    lib.attn_set_task_order.restype = i
    lib.attn_version.argtypes = []
    lib.attn_version.restype = ctypes.c_char_p
    lib.attn_probe_mma.argtypes = [i, i, i, i, vp, vp]
    lib.attn_probe_mma.restype = i
    lib.attn_probe_ex2.argtypes = [i, vp, vp, vp]
    lib.attn_probe_ex2.restype = i
    lib.attn_probe_tma.argtypes = [vp, ctypes.c_longlong, i, i, i, vp, vp]
    lib.attn_probe_tma.restype = i
    _lib = lib
    return lib


def attn_last_error() -> str:
    return load().attn_last_error().decode()


def attn_version() -> str:
    return load().attn_version().decode()


def _check(code: int):
    if code != GQA_OK:
        raise AttnError(code, attn_last_error())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dims(q, k, v=None):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, T, H, d]")
    B, T, Hq, d = q.shape
    Bk, Tk, Hkv, dk = k.shape
    if (Bk, Tk, dk) != (B, T, d):
        raise ValueError(f"k {tuple(k.shape)} does not match q {tuple(q.shape)} in B, T or d")
    if v is not None and tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"v {tuple(v.shape)} must have the shape of k {tuple(k.shape)}")
    return B, T, Hq, Hkv, d


def _args(*specs):
    """Tensor arguments (name, tensor, shape, dtype[, contiguous]), checked before their
    pointers reach the library (the C ABI takes raw pointers and cannot see sizes, types
    or devices): shapes, types and layouts of all of them first, then their devices."""
    import torch
    for spec in specs:
        name, t, shape, dtype = spec[:4]
        if t is None:
            raise ValueError(f"{name} is missing")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if (spec[4] if len(spec) > 4 else True) and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t, *_ in specs:
        if not t.is_cuda or t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name} must be on the current CUDA device, got {t.device}")


def _arg(name, t, shape, dtype, contiguous=True):
    _args((name, t, shape, dtype, contiguous))
    return t


def _ws_bytes(workspace):
    return workspace.numel() * workspace.element_size()


def _workspace(workspace, B, T, Hq, device):
    import torch
    need = attn_bwd_workspace_bytes(B, T, Hq)
    if workspace is None:
        return torch.empty(need, dtype=torch.uint8, device=device)
    if not workspace.is_contiguous() or not workspace.is_cuda or workspace.device != device:
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    if _ws_bytes(workspace) < need:
        raise ValueError(f"workspace holds {_ws_bytes(workspace)} bytes, {need} needed")
    return workspace


def _bf16():
    import torch
    return torch.bfloat16


def _f32():
    import torch
    return torch.float32


def attn_fwd(q, k, v, causal: bool = True, o=None, lse=None, stream=None):
    """O, LSE = attention(q, k, v). q [B,T,Hq,d], k/v [B,T,Hkv,d] bf16 CUDA tensors, contiguous.

    Returns (o bf16 [B,T,Hq,d], lse fp32 [B,Hq,T]). Output buffers may be passed in.
    """
    import torch
    lib = load()
    B, T, Hq, Hkv, d = _dims(q, k, v)
    _args(("q", q, q.shape, _bf16()), ("k", k, k.shape, _bf16()), ("v", v, k.shape, _bf16()))
    o = torch.empty_like(q) if o is None else _arg("o", o, q.shape, _bf16())
    lse = (torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None
           else _arg("lse", lse, (B, Hq, T), _f32()))
    _check(lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, Hq, Hkv, d, int(bool(causal)),
                        _stream_handle(stream)))
    return o, lse


def view_of(t, name: str = "tensor") -> GqaView:
    """The gqa_view_t of a bf16 CUDA tensor [B, T, H, d] whose heads are packed
    (stride(3) == 1, stride(2) == d); token and batch strides are passed as they are."""
    import torch
    if t.dim() != 4 or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise ValueError(f"{name} must be a bf16 CUDA tensor [B, T, H, d]")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} must be on the current CUDA device, got {t.device}")
    B, T, H, d = t.shape
    if t.stride(3) != 1 or (H > 1 and t.stride(2) != d):
        raise ValueError(f"{name}: the heads of a token must be packed (strides {tuple(t.stride())})")
    return GqaView(t.data_ptr(), t.stride(1), t.stride(0))


def _views(B, T, Hq, Hkv, d, extra=(), **named):
    """gqa_view_t of each named view after checking its shape ([B,T,Hq,d] for q-shaped
    names, [B,T,Hkv,d] for k-shaped ones), together with the extra argument specs."""
    _args(*((name, t, (B, T, Hkv if name in ("k", "v", "dk", "dv", "k_rot") else Hq, d), _bf16(), False)
            for name, t in named.items()), *extra)
    return [view_of(t, name) for name, t in named.items()]


def attn_fwd_strided(q, k, v, o, causal: bool = True, lse=None, stream=None):
    """attn_fwd over strided views, e.g. q, k, v sliced out of one fused [B, T, Hq+2*Hkv, d]
    projection; o (a view too) is written in place. Returns (o, lse)."""
    import torch
    lib = load()
    B, T, Hq, Hkv, d = _dims(q, k, v)
    views = _views(B, T, Hq, Hkv, d, extra=() if lse is None else (("lse", lse, (B, Hq, T), _f32()),),
                   q=q, k=k, v=v, o=o)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    _check(lib.attn_fwd_strided(*views, _ptr(lse), B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))
    return o, lse


def attn_bwd_strided(q, k, v, o, lse, dout, dq, dk, dv, causal: bool = True, workspace=None, stream=None):
    """attn_bwd over strided views; dq, dk, dv (views too, e.g. of one fused gradient
    buffer) are written in place. Returns (dq, dk, dv)."""
    lib = load()
    B, T, Hq, Hkv, d = _dims(q, k, v)
    vq, vk, vv, vo, vdo, vdq, vdk, vdv = _views(B, T, Hq, Hkv, d, extra=(("lse", lse, (B, Hq, T), _f32()),),
                                                q=q, k=k, v=v, o=o, dO=dout, dq=dq, dk=dk, dv=dv)
    workspace = _workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd_strided(vq, vk, vv, vo, _ptr(lse), vdo, vdq, vdk, vdv, _ptr(workspace), _ws_bytes(workspace),
                                B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))
    return dq, dk, dv


def attn_rope_table(T: int, d: int, base: float = 10000.0, device=None, stream=None):
    """fp32 [T, d/2, 2] table of (cos, sin) of the rotary angles t * base**(-2i/d)."""
    import torch
    lib = load()
    n = int(lib.attn_rope_table_bytes(T, d))
    if n == 0:
        raise ValueError(f"bad rotary table shape (T={T}, d={d})")
    table = torch.empty((T, d // 2, 2), dtype=torch.float32, device=device or torch.device("cuda"))
    _check(lib.attn_rope_table(_ptr(table), T, d, float(base), _stream_handle(stream)))
    return table


def attn_rope(x, table, y=None, inverse: bool = False, stream=None):
    """Rotary embedding of the bf16 view x [B, T, H, d] into y (default: in place).
    ``inverse`` rotates back, which is also the gradient of the rotation."""
    lib = load()
    if y is None:
        y = x
    if x.dim() != 4:
        raise ValueError("x must be [B, T, H, d]")
    B, T, H, d = x.shape
    if table.dim() != 3 or table.shape[0] < T or tuple(table.shape[1:]) != (d // 2, 2):
        raise ValueError(f"table {tuple(table.shape)} does not cover T={T}, d={d}")
    _args(("x", x, x.shape, _bf16(), False), ("y", y, x.shape, _bf16(), False), ("table", table, table.shape, _f32()))
    _check(lib.attn_rope(view_of(x, "x"), view_of(y, "y"), _ptr(table), B, T, H, d, int(bool(inverse)),
                         _stream_handle(stream)))
    return y


def attn_fwd_rope(q, k, v, base: float = 10000.0, causal: bool = True, o=None, lse=None, q_rot=None, k_rot=None,
                  stream=None):
    """Attention of the rotated q and k with the rotation fused in: q and k are the
    unrotated projections (views allowed), rotated by angle t * base**(-2i/d) of pair i
    of token t. Returns (o, lse, q_rot, k_rot); q_rot and k_rot (new tensors unless
    given; q_rot=q / k_rot=k rotates in place) feed attn_bwd_rope."""
    import torch
    lib = load()
    B, T, Hq, Hkv, d = _dims(q, k, v)
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device) if o is None else o
    q_rot = torch.empty(q.shape, dtype=q.dtype, device=q.device) if q_rot is None else q_rot
    k_rot = torch.empty(k.shape, dtype=k.dtype, device=k.device) if k_rot is None else k_rot
    extra = () if lse is None else (("lse", lse, (B, Hq, T), _f32()),)
    vq, vk, vv, vo, vqr, vkr = _views(B, T, Hq, Hkv, d, extra=extra, q=q, k=k, v=v, o=o, q_rot=q_rot, k_rot=k_rot)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    _check(lib.attn_fwd_rope(vq, vk, vv, vo, _ptr(lse), vqr, vkr, float(base), B, T, Hq, Hkv, d, int(bool(causal)),
                             _stream_handle(stream)))
    return o, lse, q_rot, k_rot


def attn_bwd_rope(q_rot, k_rot, v, o, lse, dout, base: float = 10000.0, causal: bool = True, dq=None, dk=None,
                  dv=None, workspace=None, stream=None):
    """Gradients of the UNROTATED q and k (and of v) from attn_fwd_rope's outputs (same
    base); the inverse rotation runs in the backward kernel's epilogue. Returns (dq, dk, dv)."""
    import torch
    lib = load()
    B, T, Hq, Hkv, d = _dims(q_rot, k_rot, v)
    dq = torch.empty(q_rot.shape, dtype=q_rot.dtype, device=q_rot.device) if dq is None else dq
    dk = torch.empty(k_rot.shape, dtype=k_rot.dtype, device=k_rot.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, device=v.device) if dv is None else dv
    vq, vk, vv, vo, vdo, vdq, vdk, vdv = _views(B, T, Hq, Hkv, d, extra=(("lse", lse, (B, Hq, T), _f32()),),
                                                q=q_rot, k=k_rot, v=v, o=o, dO=dout, dq=dq, dk=dk, dv=dv)
    workspace = _workspace(workspace, B, T, Hq, q_rot.device)
    _check(lib.attn_bwd_rope(vq, vk, vv, vo, _ptr(lse), vdo, vdq, vdk, vdv, float(base), _ptr(workspace),
                             _ws_bytes(workspace), B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))
    return dq, dk, dv


def attn_naive_workspace_bytes(B: int, T: int, Hq: int) -> int:
    return int(load().attn_naive_workspace_bytes(B, T, Hq))


def _naive_workspace(workspace, B, T, Hq, device):
    import torch
    need = attn_naive_workspace_bytes(B, T, Hq)
    if workspace is None:
        return torch.empty(need, dtype=torch.uint8, device=device)
    if not workspace.is_contiguous() or not workspace.is_cuda or workspace.device != device:
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    if _ws_bytes(workspace) < need:
        raise ValueError(f"workspace holds {_ws_bytes(workspace)} bytes, {need} needed")
    return workspace


def attn_fwd_naive(q, k, v, causal: bool = True, o=None, lse=None, workspace=None, stream=None):
    """attn_fwd by the plain kernels that write the whole score matrix (the check of the
    flash kernels). Needs attn_naive_workspace_bytes(B, T, Hq) bytes of scratch."""
    import torch
    lib = load()
    B, T, Hq, Hkv, d = _dims(q, k, v)
    _args(("q", q, q.shape, _bf16()), ("k", k, k.shape, _bf16()), ("v", v, k.shape, _bf16()))
    o = torch.empty_like(q) if o is None else _arg("o", o, q.shape, _bf16())
    lse = (torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None
           else _arg("lse", lse, (B, Hq, T), _f32()))
    workspace = _naive_workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_fwd_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace), _ws_bytes(workspace),
                              B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))
    return o, lse


def attn_bwd_naive(q, k, v, o, lse, dout, causal: bool = True, dq=None, dk=None, dv=None, workspace=None,
                   stream=None):
    """attn_bwd by the plain kernels that write the whole score matrix."""
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, o=o, lse=lse)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    workspace = _naive_workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(workspace), _ws_bytes(workspace), B, T, Hq, Hkv, d, int(bool(causal)),
                              _stream_handle(stream)))
    return dq, dk, dv


def attn_bwd_workspace_bytes(B: int, T: int, Hq: int) -> int:
    return int(load().attn_bwd_workspace_bytes(B, T, Hq))


def _bwd_inputs(q, k, v, dout, o=None, lse=None, outputs=()):
    """Checks the backward's inputs (and o, lse, and the given (name, tensor, like) outputs)."""
    B, T, Hq, Hkv, d = _dims(q, k, v)
    specs = [("q", q, q.shape, _bf16()), ("k", k, k.shape, _bf16()), ("v", v, k.shape, _bf16()),
             ("dO", dout, q.shape, _bf16())]
    if o is not None:
        specs.append(("o", o, q.shape, _bf16()))
    if lse is not None:
        specs.append(("lse", lse, (B, Hq, T), _f32()))
    specs += [(name, t, like.shape, _bf16()) for name, t, like in outputs]
    _args(*specs)
    return B, T, Hq, Hkv, d


def _grads(q, k, dq, dk, dv, need_dq=True, need_dkv=True):
    import torch
    if need_dq:
        dq = torch.empty_like(q) if dq is None else _arg("dq", dq, q.shape, _bf16())
    if need_dkv:
        dk = torch.empty_like(k) if dk is None else _arg("dk", dk, k.shape, _bf16())
        dv = torch.empty_like(k) if dv is None else _arg("dv", dv, k.shape, _bf16())
    return dq, dk, dv


def attn_bwd(q, k, v, o, lse, dout, causal: bool = True, dq=None, dk=None, dv=None, workspace=None,
             stream=None):
    """dQ, dK, dV of sum(O * dO). Returns (dq, dk, dv) bf16 with the shapes of q, k, v."""
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, o=o, lse=lse)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    workspace = _workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        _ptr(workspace), _ws_bytes(workspace), B, T, Hq, Hkv, d, int(bool(causal)),
                        _stream_handle(stream)))
    return dq, dk, dv


def attn_bwd_preprocess(o, lse, dout, workspace, stream=None):
    """Stage 1 of attn_bwd: workspace <- rowsum(dO * O) and LSE * log2(e)."""
    lib = load()
    if o.dim() != 4:
        raise ValueError("o must be [B, T, Hq, d]")
    B, T, Hq, d = o.shape
    _args(("o", o, o.shape, _bf16()), ("dO", dout, o.shape, _bf16()), ("lse", lse, (B, Hq, T), _f32()))
    workspace = _workspace(workspace, B, T, Hq, o.device)
    _check(lib.attn_bwd_preprocess(_ptr(o), _ptr(lse), _ptr(dout), _ptr(workspace), _ws_bytes(workspace), B, T,
                                   Hq, d, _stream_handle(stream)))


def attn_bwd_dq(q, k, v, dout, dq, workspace, causal: bool = True, stream=None):
    """Stage 2 of attn_bwd: dq, one task per query tile."""
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, outputs=(("dq", dq, q),))
    workspace = _workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(workspace), _ws_bytes(workspace),
                           B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))


def attn_bwd_dkv(q, k, v, dout, dk, dv, workspace, causal: bool = True, stream=None):
    """Stage 3 of attn_bwd: dk and dv, one task per key tile looping over the kv head's query heads."""
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, outputs=(("dk", dk, k), ("dv", dv, k)))
    workspace = _workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd_dkv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk), _ptr(dv), _ptr(workspace),
                            _ws_bytes(workspace), B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))


def attn_bwd_dq_dkv(q, k, v, dout, dq, dk, dv, workspace, causal: bool = True, stream=None):
    """Stages 2+3 of attn_bwd in one launch: dq, dk and dv (heaviest tasks first)."""
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, outputs=(("dq", dq, q), ("dk", dk, k), ("dv", dv, k)))
    workspace = _workspace(workspace, B, T, Hq, q.device)
    _check(lib.attn_bwd_dq_dkv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                               _ws_bytes(workspace), B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))


def attn_bwd_noalloc(q, k, v, o, lse, dout, causal: bool = True, dq=None, dk=None, dv=None, stream=None):
    """attn_bwd whose scratch is the library's own fixed device array (no workspace argument).

    For callers that may not allocate device memory where they run the backward.
    Problems needing more than NOALLOC_SCRATCH_BYTES of scratch are rejected;
    calls that overlap on one GPU race on the shared array.
    """
    lib = load()
    B, T, Hq, Hkv, d = _bwd_inputs(q, k, v, dout, o=o, lse=lse)
    dq, dk, dv = _grads(q, k, dq, dk, dv)
    _check(lib.attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, T, Hq, Hkv, d, int(bool(causal)), _stream_handle(stream)))
    return dq, dk, dv


def attn_sync_status(stream=None) -> int:
    """Synchronise the stream and return the device status code (0 = OK, 4 = a wait timed out)."""
    return int(load().attn_sync_status(_stream_handle(stream)))


def attn_selftest_timeout(budget_ns: int, stream=None):
    _check(load().attn_selftest_timeout(int(budget_ns), _stream_handle(stream)))


def attn_set_task_order(order: int):
    """Backward task order: 0 by size (default), 1 tile-major, 2 group-major. The
    results are the same bits in any order; this only moves the time."""
    _check(load().attn_set_task_order(int(order)))


def attn_set_wait_budget_ns(budget_ns: int):
    load().attn_set_wait_budget_ns(int(budget_ns))


def probe_rates(iters: int = 4096, device=None):
    """Measured rates of this GPU's units, one CTA per SM (attn_probe_mma, attn_probe_ex2):
    tcgen05 bf16 MMA FLOP/cycle/SM for N = 64, 128, 256 with A in shared or tensor
    memory, into one accumulator or alternately into two, ex2 lanes/cycle/SM, and the
    SM clock seen during the MMA probes (MHz, median over SMs). Returns a dict; the
    medians over SMs are reported."""
    import statistics
    import torch
    lib = load()
    dev = device or torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.zeros((sms, 2), dtype=torch.int64, device=dev)
    res = {"sms": sms, "mma": {}}
    clocks = []
    for chains in (1, 2):
        for a_tmem in (0, 1):
            for n in (64, 128, 256):
                if chains == 2 and a_tmem and n == 256:
                    continue
                _check(lib.attn_probe_mma(n, a_tmem, chains, iters, _ptr(out), _stream_handle(None)))
                _check(attn_sync_status())
                rec = out.cpu().tolist()
                flop = iters * 4 * 2.0 * 128 * n * 16
                rate = statistics.median(flop / c for c, _ in rec)
                clocks += [c / t * 1e3 for c, t in rec]
                res["mma"][f"{'ts' if a_tmem else 'ss'}_n{n}_{'one' if chains == 1 else 'two'}_acc"] = rate
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    sink = torch.zeros(4, dtype=torch.float32, device=dev)
    _check(lib.attn_probe_ex2(iters, _ptr(cyc), _ptr(sink), _stream_handle(None)))
    _check(attn_sync_status())
    res["ex2_lanes_per_clk"] = statistics.median(1024 * 8 * iters / c for c in cyc.cpu().tolist())
    res["sm_mhz_during_mma"] = statistics.median(clocks)
    best = max(res["mma"].values())
    res["mma_peak_tflops_at_probe_clock"] = best * sms * res["sm_mhz_during_mma"] * 1e6 / 1e12
    return res


def probe_tma(sizes_mb=(32, 2048), stages: int = 6, ctas_per_sm=(1, 2), iters: int = 2000, device=None):
    """Measured rate of the TMA path that fills the kernels' operand rings
    (attn_probe_tma): 16 KB tiles into shared memory, `stages` requests in flight per
    CTA, one or two CTAs per SM, over a buffer of each size in MB (32 MB fits the L2,
    2048 MB does not). Returns a list of dicts: TB/s over the slowest CTA and the
    implied load latency in microseconds (bytes in flight per SM over the per-SM
    rate)."""
    import torch
    lib = load()
    dev = device or torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = []
    for mb in sizes_mb:
        buf = torch.zeros(int(mb) << 20, dtype=torch.uint8, device=dev)
        for cps in ctas_per_sm:
            st = min(stages, 8 if cps == 1 else 6)
            out = torch.zeros(sms * cps, dtype=torch.int64, device=dev)
            for _ in range(2):  # the first call warms the caches and the clocks
                _check(lib.attn_probe_tma(_ptr(buf), buf.numel(), st, cps, iters, _ptr(out), _stream_handle(None)))
                _check(attn_sync_status())
            ns = max(out.cpu().tolist())
            rate = sms * cps * iters * 16384 / ns * 1e9  # bytes/s
            latency_us = st * cps * 16384 / (rate / sms) * 1e6
            res.append({"buffer_mb": mb, "ctas_per_sm": cps, "stages": st, "tbps": rate / 1e12,
                        "latency_us": latency_us})
        del buf
    return res
