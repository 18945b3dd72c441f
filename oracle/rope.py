"""Oracle: rotary position embedding applied to Q and K before attention, f64.

TEST INFRASTRUCTURE, like the rest of ``oracle/``.

The pages list RoPE with GQA attention as one of the transformer block's ops,
forward and backward (tang page, "A transformer": "RMSNorm, RoPE, GQA
attention, SwiGLU"; RustingBrain docs, "What is in the box": rotary
positions), but print no formula. Reading: the rotary position embedding in
its rotate-half pairing. With caller-supplied tables cos, sin of shape
[S, D/2] (entry [p, i] for position p and frequency i), each query or key row
x at position p becomes

    x'[i]       = x[i] cos[p, i] - x[i + D/2] sin[p, i]
    x'[i + D/2] = x[i + D/2] cos[p, i] + x[i] sin[p, i]      (0 <= i < D/2),

a rotation of the plane (x[i], x[i + D/2]) by the angle whose cosine and sine
the tables hold. Attention then runs on the rotated Q and K; V is not rotated.
The gradient with respect to the unrotated input is the rotated gradient
turned back by the transposed rotation (the same formula with -sin).
"""

from __future__ import annotations

import numpy as np

from .attention import backward, forward


def rotate(x, cos, sin):
    """x [..., S, D] rotated per position: rows p use cos[p], sin[p] ([S, D/2])."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)
    s = np.asarray(sin, dtype=np.float64)
    h = x.shape[-1] // 2
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def unrotate(g, cos, sin):
    """The transposed rotation: the gradient with respect to x from the gradient with respect to rotate(x)."""
    return rotate(g, cos, -np.asarray(sin, dtype=np.float64))


def forward_rope(q, k, v, cos, sin, causal: bool = True, scale: float | None = None):
    """O, LSE of attention over rotate(q), rotate(k), v (layouts as ``oracle.attention.forward``)."""
    return forward(rotate(q, cos, sin), rotate(k, cos, sin), v, causal=causal, scale=scale)


def backward_rope(q, k, v, dO, cos, sin, causal: bool = True, scale: float | None = None):
    """dQ, dK, dV of L = sum(O * dO) with respect to the unrotated q, k (and v)."""
    gq, gk, gv = backward(rotate(q, cos, sin), rotate(k, cos, sin), v, dO, causal=causal, scale=scale)
    return unrotate(gq, cos, sin), unrotate(gk, cos, sin), gv
