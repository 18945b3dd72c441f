"""Oracle: attention of a few new queries against a key/value cache, f64 (decode / prefill over a cache).

TEST INFRASTRUCTURE, like the rest of ``oracle/``.

The KV-cached decoding of the RustingBrain docs ("Training infrastructure",
"KV-cached decoding") and the decode step of the tang page ("An LLM") attend
Sq new query rows to Sk >= Sq cached keys. Reading (the pages give no
formula): the new queries are the last Sq positions of the sequence, so
query i (0-based among the new ones) sits at absolute position Sk - Sq + i
and, when causal, sees keys j <= Sk - Sq + i (bottom-right alignment; for
Sq = Sk this is the ordinary causal mask). Otherwise the definition is that
of ``oracle.attention.forward``, evaluated row by row.
"""

from __future__ import annotations

import numpy as np

from .attention import _softmax_stats, kv_head_of, scores


def forward_cached(q, k_cache, v_cache, causal: bool = True, scale: float | None = None):
    """O [B, Hq, Sq, D] and LSE [B, Hq, Sq] (f64) of q [B, Hq, Sq, D] against k/v [B, Hkv, Sk, D]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_cache, dtype=np.float64)
    v = np.asarray(v_cache, dtype=np.float64)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    assert k.shape == (B, Hkv, Sk, D) and v.shape == k.shape and Hq % Hkv == 0 and Sq <= Sk
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    rows = (Sk - Sq) + np.arange(Sq)
    O = np.zeros((B, Hq, Sq, D))
    L = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            s = scores(q[b, h], k[b, g], rows, causal, scale)
            lse, p = _softmax_stats(s)
            O[b, h] = p @ v[b, g]
            L[b, h] = lse
    return O, L
