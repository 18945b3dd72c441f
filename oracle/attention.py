"""Oracle: causal grouped-query attention, forward and backward, by its plain definition in f64.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. It shares no code
with the CUDA library and imports nothing from it.

What is computed (tang, "How tang works" section 3, "Optimizations are
derived, not written", equations (5)-(6): attention as written, scores
stored, a row max and two sums; the derived flash form gives "the same
answer"). Grouped-query heads follow "GQA 12/4 heads" / ``.heads(8, 2, 64)``
of the RustingBrain docs ("Where it stands against PyTorch and TensorFlow";
"A language model in twenty lines"). The backward follows the reading that
a gradient through the comprehension is itself a comprehension with no
intermediate tensors (aiinsiders.net, "A compiler that derives GPU kernels
matches hand-tuned code"), evaluated here in the plain, materialised form.

Readings where the pages are silent (all of them listed in the design notes):

* layout BHSD: q, dO, O, dQ are [B, Hq, S, D]; k, v, dK, dV are [B, Hkv, S, D];
  LSE is [B, Hq, S];
* query head h reads KV head h // (Hq // Hkv) (grouped-contiguous heads);
* causal means key j is visible to query i iff j <= i (Sq = Sk = S);
* scale multiplies the scores before the softmax; LSE is the natural-log
  log-sum-exp of the scaled scores;
* the backward is the gradient of L = sum(O * dO) for the given dO.

Every input is widened exactly to float64 before any arithmetic; every
result is float64. Rows are independent in the definition, so functions
that take a ``rows`` argument evaluate the same definition on a subset of
query (or key) rows; nothing is blocked, fused or reordered within a row.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "kv_head_of",
    "scores",
    "forward",
    "forward_rows",
    "backward",
    "backward_dq_rows",
    "backward_dkdv_rows",
]


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """Query head h reads KV head floor(h / G), G = Hq / Hkv."""
    return h // (Hq // Hkv)


def _check(q, k, v):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, S, D = q.shape
    assert k.shape[0] == B and k.shape[2] == S and k.shape[3] == D, (q.shape, k.shape)
    assert v.shape == k.shape, (k.shape, v.shape)
    Hkv = k.shape[1]
    assert Hq % Hkv == 0, (Hq, Hkv)
    return q, k, v, B, Hq, Hkv, S, D


def scores(q_rows, k_head, row_idx, causal: bool, scale: float):
    """s_ij = scale * q_i . k_j, with -inf where key j is not visible to query i.

    q_rows: [n, D] query rows with absolute positions ``row_idx``;
    k_head: [S, D] all keys of the KV head. Returns [n, S].
    """
    s = scale * (q_rows @ k_head.T)
    if causal:
        j = np.arange(k_head.shape[0])[None, :]
        s = np.where(j <= np.asarray(row_idx)[:, None], s, -np.inf)
    return s


def _softmax_stats(s):
    """Row max m, LSE = m + ln sum exp(s - m), and P = exp(s - LSE) (masked entries give 0)."""
    m = s.max(axis=1)
    lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return lse, p


def forward_rows(q, k, v, b: int, h: int, rows, causal: bool, scale: float):
    """O and LSE of query head h of batch b at the query rows ``rows`` (absolute indices).

    Returns (O [n, D], LSE [n]) in float64.
    """
    q, k, v, B, Hq, Hkv, S, D = _check(q, k, v)
    rows = np.asarray(rows, dtype=np.int64)
    g = kv_head_of(h, Hq, Hkv)
    s = scores(q[b, h, rows], k[b, g], rows, causal, scale)
    lse, p = _softmax_stats(s)
    return p @ v[b, g], lse


def forward(q, k, v, causal: bool = True, scale: float | None = None, row_block: int = 2048):
    """Full forward: O [B, Hq, S, D] and LSE [B, Hq, S], float64.

    Evaluates ``forward_rows`` on every row (in row blocks of ``row_block``
    so that the score rows of one block, not S x S, are held at once).
    """
    q, k, v, B, Hq, Hkv, S, D = _check(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.zeros((B, Hq, S, D))
    LSE = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            for r0 in range(0, S, row_block):
                rows = np.arange(r0, min(S, r0 + row_block))
                O[b, h, rows], LSE[b, h, rows] = forward_rows(q, k, v, b, h, rows, causal, scale)
    return O, LSE


def backward(q, k, v, dO, causal: bool = True, scale: float | None = None):
    """Gradients (dQ, dK, dV) of L = sum(O * dO), float64, by the materialised definition.

    Per (b, h), with g = kv_head_of(h):
      P = softmax(scale * q k^T + mask), O = P v,
      dP = dO v^T, D_i = sum_d dO_id O_id, dS = P * (dP - D),
      dQ = scale * dS k,  dK[g] += scale * dS^T q,  dV[g] += P^T dO.
    dK and dV of a KV head are summed over the query heads that read it.
    """
    q, k, v, B, Hq, Hkv, S, D = _check(q, k, v)
    dO = np.asarray(dO, dtype=np.float64)
    assert dO.shape == q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    rows = np.arange(S)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            s = scores(q[b, h], k[b, g], rows, causal, scale)
            _, P = _softmax_stats(s)
            O = P @ v[b, g]
            dP = dO[b, h] @ v[b, g].T
            Dvec = (dO[b, h] * O).sum(axis=1)
            dS = P * (dP - Dvec[:, None])
            dQ[b, h] = scale * (dS @ k[b, g])
            dK[b, g] += scale * (dS.T @ q[b, h])
            dV[b, g] += P.T @ dO[b, h]
    return dQ, dK, dV


def backward_dq_rows(q, k, v, dO, b: int, h: int, rows, causal: bool, scale: float):
    """dQ of query head h of batch b at query rows ``rows`` ([n, D], float64).

    Row i of dQ needs only row i of P, dP and D, so this is ``backward``
    restricted to those rows.
    """
    q, k, v, B, Hq, Hkv, S, D = _check(q, k, v)
    dO = np.asarray(dO, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    g = kv_head_of(h, Hq, Hkv)
    s = scores(q[b, h, rows], k[b, g], rows, causal, scale)
    _, P = _softmax_stats(s)
    O = P @ v[b, g]
    dP = dO[b, h, rows] @ v[b, g].T
    Dvec = (dO[b, h, rows] * O).sum(axis=1)
    dS = P * (dP - Dvec[:, None])
    return scale * (dS @ k[b, g])


def backward_dkdv_rows(q, k, v, dO, b: int, g: int, kv_rows, causal: bool, scale: float,
                       row_block: int = 1024):
    """dK and dV of KV head g of batch b at key rows ``kv_rows`` ([n, D] each, float64).

    Column j of dS needs, for every query row i of every query head of the
    group, row i's LSE and D_i, so every query row that can see key j is
    evaluated (in row blocks); only the columns ``kv_rows`` of P and dS are
    kept. Summed over the query heads h with kv_head_of(h) == g.
    """
    q, k, v, B, Hq, Hkv, S, D = _check(q, k, v)
    dO = np.asarray(dO, dtype=np.float64)
    J = np.asarray(kv_rows, dtype=np.int64)
    G = Hq // Hkv
    dK = np.zeros((len(J), D))
    dV = np.zeros((len(J), D))
    first = int(J.min()) if causal else 0
    for h in range(g * G, (g + 1) * G):
        for r0 in range(first, S, row_block):
            rows = np.arange(r0, min(S, r0 + row_block))
            s = scores(q[b, h, rows], k[b, g], rows, causal, scale)
            _, P = _softmax_stats(s)
            O = P @ v[b, g]
            Dvec = (dO[b, h, rows] * O).sum(axis=1)
            PJ = P[:, J]
            dPJ = dO[b, h, rows] @ v[b, g, J].T
            dSJ = PJ * (dPJ - Dvec[:, None])
            dK += scale * (dSJ.T @ q[b, h, rows])
            dV += PJ.T @ dO[b, h, rows]
    return dK, dV
