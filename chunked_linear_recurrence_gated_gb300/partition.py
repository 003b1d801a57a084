"""Chunk boundaries for splitting one long sequence into N chunks.

Host utility for the hybrid cost model of the StateFlow review ("What carries
the argument": Cost_i = (L_lin C_lin + C_dense) s_i + L_soft C_soft
(c_i s_i + s_i^2 / 2), Eq. 9; the family c_i(alpha) = (1 - alpha) c_i^equal +
alpha c_i^hybrid). c_i is read as the start offset of chunk i (the prefix
length its softmax layers attend to), so the cumulative cost up to offset x is
f(x) = a x + b x^2 / 2 with a = L_lin C_lin + C_dense, b = L_soft C_soft, and
the equal-cost boundaries solve f(x_i) = i f(T) / N. Both the equal-length and
the equal-cost boundaries are linear in the offsets, so blending boundaries
with alpha is the same as blending lengths. Boundaries are rounded half-up to
a multiple of `multiple` (64 keeps every chunk start on a kernel block edge).
"""
from __future__ import annotations

import math


def hybrid_boundaries(T: int, N: int, alpha: float, L_lin: float = 3.0, L_soft: float = 1.0,
                      C_lin: float = 1.0, C_dense: float = 1.0, C_soft: float = 1.0,
                      multiple: int = 64) -> list[int]:
    """Return N + 1 increasing boundaries [0, ..., T]."""
    if N < 1 or T < N * multiple:
        raise ValueError("need T >= N * multiple")
    a = L_lin * C_lin + C_dense
    b = L_soft * C_soft
    fT = a * T + b * T * T / 2.0
    out = [0]
    for i in range(1, N):
        target = i * fT / N
        if b > 0:
            x_h = (-a + math.sqrt(a * a + 2.0 * b * target)) / b
        else:
            x_h = target / a
        x_e = i * T / N
        x = (1.0 - alpha) * x_e + alpha * x_h
        r = int(math.floor(x / multiple + 0.5)) * multiple
        r = min(max(r, out[-1] + multiple), T - (N - i) * multiple)
        out.append(r)
    out.append(T)
    return out
