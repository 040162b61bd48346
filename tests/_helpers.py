"""Shared helpers for the GPU parity tests (comparison metrics and guard buffers)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the GPU path against the f64 oracle:
#  O: max |gpu - oracle| over all elements; LSE: max abs; dQ/dK/dV: ||gpu - oracle||_F / ||oracle||_F.
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD = 1e-2


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def max_abs(a, r) -> float:
    return float(np.max(np.abs(a - r))) if a.size else 0.0


def half_ulp_bf16(r: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |r| (8 significant bits): the rounding error any bf16 output may carry."""
    mag = np.maximum(np.abs(r), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(mag)).astype(np.int64) - 8)


def o_err(a, r) -> float:
    """O error beyond the bf16 output's own rounding: max(|a - r| - half_ulp_bf16(r)).

    For |O| in [4, 8) a bf16 value is only known to +-2^-6 = 0.0156, so a plain
    max-abs bound of 1e-2 is unattainable by any bf16 output there; the O
    tolerance applies to the error the computation adds on top of that.
    """
    return float(np.max(np.abs(a - r) - half_ulp_bf16(r))) if a.size else 0.0


def rel_fro(a, r) -> float:
    n = np.linalg.norm(r)
    return float(np.linalg.norm(a - r) / n) if n > 0 else float(np.linalg.norm(a))


def worst_index(a, r):
    """(index tuple, gpu value, oracle value) of the largest absolute difference."""
    idx = np.unravel_index(np.argmax(np.abs(a - r)), a.shape)
    return tuple(int(i) for i in idx), float(a[idx]), float(r[idx])


GUARD = 4096  # bytes of guard on each side of a guarded output


class Guarded:
    """A CUDA tensor embedded in a larger buffer whose edges hold a known byte pattern."""

    def __init__(self, shape, dtype, device):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.empty(n + 2 * GUARD, dtype=torch.uint8, device=device)
        self.raw.fill_(0xA5)
        self.tensor = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        self.n = n

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool((head == 0xA5).all().item()) and bool((tail == 0xA5).all().item())


def check_against_oracle(out, ref, label):
    o, lse = f64(out["o"]), f64(out["lse"])
    e_o, e_l = o_err(o, ref["o"]), max_abs(lse, ref["lse"])
    raw_o = max_abs(o, ref["o"])
    e_dq = rel_fro(f64(out["dq"]), ref["dq"])
    e_dk = rel_fro(f64(out["dk"]), ref["dk"])
    e_dv = rel_fro(f64(out["dv"]), ref["dv"])
    msg = (f"{label}: O {e_o:.2e} beyond bf16 half-ulp (raw {raw_o:.2e}, worst {worst_index(o, ref['o'])}), LSE {e_l:.2e} "
           f"(worst {worst_index(lse, ref['lse'])}), dQ {e_dq:.2e} dK {e_dk:.2e} dV {e_dv:.2e}")
    print(msg)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), msg
    assert e_o <= TOL_O and e_l <= TOL_LSE, msg
    assert e_dq <= TOL_GRAD and e_dk <= TOL_GRAD and e_dv <= TOL_GRAD, msg
