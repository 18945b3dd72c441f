"""Oracle: attention over a batch of variable-length sequences packed along the token axis, f64.

TEST INFRASTRUCTURE, like the rest of ``oracle/``.

The pages train on batches of token windows (RustingBrain docs, "Training
infrastructure": ``batch(step, 8, 512)`` windows drawn from a flat token file)
and prefill new tokens over a cache (tang page, "An LLM": prefill 512); they
give no formula for a batch whose sequences differ in length. Reading (the
plainest one consistent with the rest): the sequences of a batch are laid
end to end along the token axis, one [H, T, D] tensor per operand, with
sequence i owning rows cu_seqlens[i] .. cu_seqlens[i+1]-1; no query attends
to another sequence's keys; within sequence i, with Sq_i query rows and
Sk_i >= Sq_i key rows, query r sits at position Sk_i - Sq_i + r and (causal)
sees keys j <= Sk_i - Sq_i + r of that sequence, the alignment of
``oracle.decode.forward_cached``. So the packed result is that of each
sequence on its own, which is exactly what is computed here: every sequence
is cut out and handed to the plain definition.
"""

from __future__ import annotations

import numpy as np

from .attention import backward
from .decode import forward_cached


def _bounds(cu, T):
    cu = np.asarray(cu, dtype=np.int64)
    assert cu.ndim == 1 and cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0), (cu, T)
    return cu


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = True, scale: float | None = None):
    """O [Hq, Tq, D] and LSE [Hq, Tq] (f64) of packed queries q [Hq, Tq, D] against packed keys and
    values k, v [Hkv, Tk, D]; sequence i owns query rows cu_seqlens_q[i]:cu_seqlens_q[i+1] and key
    rows cu_seqlens_k[i]:cu_seqlens_k[i+1] (at least as many keys as queries)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, Tq, D = q.shape
    Hkv, Tk = k.shape[0], k.shape[1]
    assert k.shape == (Hkv, Tk, D) and v.shape == k.shape and Hq % Hkv == 0
    cq = _bounds(cu_seqlens_q, Tq)
    ck = _bounds(cu_seqlens_k, Tk)
    assert len(cq) == len(ck)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.zeros((Hq, Tq, D))
    L = np.zeros((Hq, Tq))
    for i in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[i], cq[i + 1], ck[i], ck[i + 1]
        if q1 == q0:
            continue
        assert q1 - q0 <= k1 - k0, "a sequence has more queries than keys"
        Oi, Li = forward_cached(q[None, :, q0:q1], k[None, :, k0:k1], v[None, :, k0:k1], causal=causal, scale=scale)
        O[:, q0:q1] = Oi[0]
        L[:, q0:q1] = Li[0]
    return O, L


def backward_varlen(q, k, v, dO, cu_seqlens, causal: bool = True, scale: float | None = None):
    """Gradients (dQ [Hq, T, D], dK, dV [Hkv, T, D]) of L = sum(O * dO), f64, for packed
    self-attention: queries and keys share the sequence bounds cu_seqlens."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    Hq, T, D = q.shape
    assert dO.shape == q.shape and k.shape[1] == T
    cu = _bounds(cu_seqlens, T)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for i in range(len(cu) - 1):
        s0, s1 = cu[i], cu[i + 1]
        if s1 == s0:
            continue
        gq, gk, gv = backward(q[None, :, s0:s1], k[None, :, s0:s1], v[None, :, s0:s1], dO[None, :, s0:s1],
                              causal=causal, scale=scale)
        dQ[:, s0:s1] = gq[0]
        dK[:, s0:s1] = gk[0]
        dV[:, s0:s1] = gv[0]
    return dQ, dK, dV
