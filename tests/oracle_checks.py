"""Checks that pin the oracle to things other than itself.

Each ``check_*`` takes an oracle-like module (``forward``, ``backward``,
``forward_rows``, ``backward_dq_rows``, ``backward_dkdv_rows``) and raises
AssertionError when the pin does not hold. The same checks run on the real
oracle (they must all pass) and on copies of it with a planted mistake (at
least one must fail), which shows that they would catch that mistake.
"""

from __future__ import annotations

import json
import math
from decimal import Decimal, localcontext
from pathlib import Path

import numpy as np
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _dyadic(rng, shape, denom=8, lo=-12, hi=12):
    """Small exactly-representable values (multiples of 1/denom)."""
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) / denom


def _relerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


# ---------------------------------------------------------------------------
# 1. Decimal brute force of the textbook form (no max subtraction needed in
#    50-digit decimal arithmetic): O_i = sum_j e^{s_ij} v_j / sum_j e^{s_ij},
#    LSE_i = ln sum_j e^{s_ij}.
# ---------------------------------------------------------------------------

def brute_forward_decimal(q, k, v, causal, scale, prec=50):
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    O = np.zeros((B, Hq, S, D))
    L = np.zeros((B, Hq, S))
    with localcontext() as ctx:
        ctx.prec = prec
        sc = Decimal(float(scale))
        for b in range(B):
            for h in range(Hq):
                g = h // G
                for i in range(S):
                    terms = []
                    for j in range(S):
                        if causal and j > i:
                            continue
                        dot = sum(Decimal(float(q[b, h, i, d])) * Decimal(float(k[b, g, j, d]))
                                  for d in range(D))
                        terms.append((j, (sc * dot).exp()))
                    Z = sum(w for _, w in terms)
                    for d in range(D):
                        num = sum(w * Decimal(float(v[b, g, j, d])) for j, w in terms)
                        O[b, h, i, d] = float(num / Z)
                    L[b, h, i] = float(Z.ln())
    return O, L


def check_decimal_bruteforce(orc):
    rng = _rng(11)
    for (B, Hq, Hkv, S, D, causal, scale) in [
        (1, 4, 2, 5, 3, True, 0.75),
        (1, 4, 2, 6, 4, False, 0.5),
        (2, 2, 1, 4, 2, True, 1.0 / math.sqrt(2.0)),
        (1, 3, 3, 3, 4, True, 0.3),
    ]:
        q = _dyadic(rng, (B, Hq, S, D))
        k = _dyadic(rng, (B, Hkv, S, D))
        v = _dyadic(rng, (B, Hkv, S, D))
        O, L = orc.forward(q, k, v, causal=causal, scale=scale)
        Ob, Lb = brute_forward_decimal(q, k, v, causal, scale)
        assert _relerr(O, Ob) <= 1e-14, ("O vs decimal", _relerr(O, Ob))
        assert np.max(np.abs(L - Lb)) <= 1e-13 * max(1.0, np.max(np.abs(Lb))), ("LSE vs decimal",)


# ---------------------------------------------------------------------------
# 2. Central finite differences of L = sum(O * dO).
# ---------------------------------------------------------------------------

def check_finite_differences(orc):
    rng = _rng(12)
    B, Hq, Hkv, S, D = 1, 4, 2, 8, 4
    for causal, scale in [(True, 0.7), (False, 1.3)]:
        q = rng.standard_normal((B, Hq, S, D))
        k = rng.standard_normal((B, Hkv, S, D))
        v = rng.standard_normal((B, Hkv, S, D))
        dO = rng.standard_normal((B, Hq, S, D))

        def loss(q_, k_, v_):
            O, _ = orc.forward(q_, k_, v_, causal=causal, scale=scale)
            return float(np.sum(O * dO))

        def loss_with(name, x_):
            return loss(x_ if name == "q" else q, x_ if name == "k" else k, x_ if name == "v" else v)

        dQ, dK, dV = orc.backward(q, k, v, dO, causal=causal, scale=scale)
        eps = 1e-5
        for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp = x.copy()
                xp[idx] += eps
                xm = x.copy()
                xm[idx] -= eps
                fd[idx] = (loss_with(name, xp) - loss_with(name, xm)) / (2 * eps)
            err = _relerr(g, fd)
            assert err <= 1e-6, (f"d{name} vs finite differences", causal, err)


# ---------------------------------------------------------------------------
# 3. Closed forms.
# ---------------------------------------------------------------------------

def check_closed_forms(orc):
    rng = _rng(13)
    B, Hq, Hkv, S, D = 2, 6, 2, 9, 5
    G = Hq // Hkv
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    dO = rng.standard_normal((B, Hq, S, D))
    q0 = np.zeros((B, Hq, S, D))
    heads = np.arange(Hq) // G
    # Q = 0, causal: O_i is the prefix mean of V, LSE_i = ln(i + 1).
    O, L = orc.forward(q0, k, v, causal=True, scale=0.9)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    assert _relerr(O, prefix_mean[:, heads]) <= 1e-13, "Q=0 prefix mean"
    assert np.max(np.abs(L - np.log(np.arange(1, S + 1))[None, None, :])) <= 1e-13, "Q=0 LSE"
    # Q = 0, non-causal: O_i is the mean of V, LSE_i = ln S.
    O, L = orc.forward(q0, k, v, causal=False, scale=0.9)
    assert _relerr(O, np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)[:, heads]) <= 1e-13
    assert np.max(np.abs(L - math.log(S))) <= 1e-13
    # Q = 0, causal: P_ij = 1 / (i + 1) for j <= i, so dV_j = sum_{h in group} sum_{i >= j} dO_{h,i} / (i + 1);
    # dK_j = scale sum_i dS_ij q_i = 0 because q = 0.
    _, dK, dV = orc.backward(q0, k, v, dO, causal=True, scale=0.9)
    w = dO / np.arange(1, S + 1)[None, None, :, None]
    suffix = np.flip(np.cumsum(np.flip(w, axis=2), axis=2), axis=2)  # sum over i >= j
    dV_ref = np.zeros_like(v)
    for h in range(Hq):
        dV_ref[:, heads[h]] += suffix[:, h]
    assert _relerr(dV, dV_ref) <= 1e-13, "Q=0 dV"
    assert np.max(np.abs(dK)) <= 1e-14, "Q=0 dK"
    # S = 1: O = v_0, LSE = scale q_0 . k_0, dQ = dK = 0, dV = sum over the group of dO.
    q1 = rng.standard_normal((B, Hq, 1, D))
    k1 = rng.standard_normal((B, Hkv, 1, D))
    v1 = rng.standard_normal((B, Hkv, 1, D))
    dO1 = rng.standard_normal((B, Hq, 1, D))
    O, L = orc.forward(q1, k1, v1, causal=True, scale=0.4)
    assert _relerr(O, v1[:, heads]) <= 1e-15
    assert np.max(np.abs(L - 0.4 * np.einsum("bhsd,bhsd->bhs", q1, k1[:, heads]))) <= 1e-14
    dQ, dK, dV = orc.backward(q1, k1, v1, dO1, causal=True, scale=0.4)
    assert np.max(np.abs(dQ)) <= 1e-14 and np.max(np.abs(dK)) <= 1e-14
    assert _relerr(dV, dO1.reshape(B, Hkv, G, 1, D).sum(axis=2)) <= 1e-14
    # Softmax rows sum to 1: with V = 1 every output is 1.
    q = rng.standard_normal((B, Hq, S, D))
    O, _ = orc.forward(q, k, np.ones_like(v), causal=True, scale=1.1)
    assert np.max(np.abs(O - 1.0)) <= 1e-14, "rows of P sum to 1"


# ---------------------------------------------------------------------------
# 4. Invariants.
# ---------------------------------------------------------------------------

def check_invariants(orc):
    rng = _rng(14)
    B, Hq, Hkv, S, D = 2, 4, 2, 10, 6
    G = Hq // Hkv
    heads = np.arange(Hq) // G
    q = rng.standard_normal((B, Hq, S, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    dO = rng.standard_normal((B, Hq, S, D))
    scale = 0.6
    for causal in (True, False):
        O, L = orc.forward(q, k, v, causal=causal, scale=scale)
        # K shift: k_j += c for every j leaves O unchanged and adds scale q_i . c to LSE_i.
        c = rng.standard_normal((B, Hkv, 1, D))
        O2, L2 = orc.forward(q, k + c, v, causal=causal, scale=scale)
        assert _relerr(O2, O) <= 1e-12, "K shift O"
        shift = scale * np.einsum("bhsd,bhd->bhs", q, c[:, heads, 0])
        assert np.max(np.abs(L2 - (L + shift))) <= 1e-12, "K shift LSE"
        # Scale folds into Q.
        O3, L3 = orc.forward(q * 2.0, k, v, causal=causal, scale=scale / 2.0)
        assert _relerr(O3, O) <= 1e-13 and np.max(np.abs(L3 - L)) <= 1e-13
        # sum_j dK_j = 0 because every row of dS sums to 0.
        dQ, dK, dV = orc.backward(q, k, v, dO, causal=causal, scale=scale)
        assert np.max(np.abs(dK.sum(axis=2))) <= 1e-12 * np.max(np.abs(dK)) * S, "sum_j dK = 0"
        # GQA equals MHA over repeated K/V, with dK/dV of the copies summed over the group.
        kr = np.repeat(k, G, axis=1)
        vr = np.repeat(v, G, axis=1)
        Om, Lm = orc.forward(q, kr, vr, causal=causal, scale=scale)
        assert _relerr(Om, O) <= 1e-14 and np.max(np.abs(Lm - L)) <= 1e-14, "GQA = MHA(repeat)"
        dQm, dKm, dVm = orc.backward(q, kr, vr, dO, causal=causal, scale=scale)
        assert _relerr(dQm, dQ) <= 1e-13
        assert _relerr(dKm.reshape(B, Hkv, G, S, D).sum(axis=2), dK) <= 1e-13
        assert _relerr(dVm.reshape(B, Hkv, G, S, D).sum(axis=2), dV) <= 1e-13
        # Rows beyond the causal prefix do not change earlier outputs (causality).
        if causal:
            q4, k4, v4 = q.copy(), k.copy(), v.copy()
            k4[:, :, -3:] += 5.0
            v4[:, :, -3:] -= 2.0
            O4, L4 = orc.forward(q4, k4, v4, causal=True, scale=scale)
            assert _relerr(O4[:, :, :-3], O[:, :, :-3]) <= 1e-15
            assert _relerr(O4[:, :, -3:], O[:, :, -3:]) > 1e-3


# ---------------------------------------------------------------------------
# 5. Library special case: torch float64 scaled_dot_product_attention (CPU)
#    on K/V repeated over the group, forward and autograd backward.
# ---------------------------------------------------------------------------

def check_torch_sdpa(orc):
    rng = _rng(15)
    for (B, Hq, Hkv, S, D, causal, scale) in [(1, 4, 2, 128, 64, True, 0.125),
                                              (2, 6, 2, 37, 16, True, 0.3),
                                              (1, 4, 4, 23, 8, False, 0.5)]:
        G = Hq // Hkv
        q = rng.standard_normal((B, Hq, S, D))
        k = rng.standard_normal((B, Hkv, S, D))
        v = rng.standard_normal((B, Hkv, S, D))
        dO = rng.standard_normal((B, Hq, S, D))
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        out = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
            is_causal=causal, scale=scale)
        out.backward(torch.tensor(dO))
        O, L = orc.forward(q, k, v, causal=causal, scale=scale)
        assert _relerr(O, out.detach().numpy()) <= 1e-12, "O vs torch SDPA"
        sc = scale * torch.einsum("bhid,bhjd->bhij", torch.tensor(q),
                                  torch.tensor(k).repeat_interleave(G, dim=1))
        if causal:
            sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        assert np.max(np.abs(L - torch.logsumexp(sc, dim=-1).numpy())) <= 1e-12, "LSE vs torch"
        dQ, dK, dV = orc.backward(q, k, v, dO, causal=causal, scale=scale)
        assert _relerr(dQ, tq.grad.numpy()) <= 1e-12, "dQ vs torch autograd"
        assert _relerr(dK, tk.grad.numpy()) <= 1e-12, "dK vs torch autograd"
        assert _relerr(dV, tv.grad.numpy()) <= 1e-12, "dV vs torch autograd"


# ---------------------------------------------------------------------------
# 6. Monoid regrouping: chunked online softmax in several groupings equals
#    the single-pass definition.
# ---------------------------------------------------------------------------

def check_monoid_regrouping(orc, monoid):
    rng = _rng(16)
    B, Hq, Hkv, S, D = 1, 2, 1, 97, 8
    scale = 0.35
    q = rng.standard_normal((B, Hq, S, D)) * 3.0  # wide score range
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    O, L = orc.forward(q, k, v, causal=True, scale=scale)
    for h in range(Hq):
        for i in (0, 1, 31, 64, 96):
            s = scale * (q[0, h, i] @ k[0, 0, : i + 1].T)
            V = v[0, 0, : i + 1]
            n = i + 1
            cuts = np.sort(rng.choice(np.arange(1, n), size=min(n - 1, 7), replace=False)) if n > 1 else []
            bounds = [0, *[int(c) for c in cuts], n]
            states = [monoid.chunk_state(s[a:b], V[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
            for st in (monoid.fold_left(states), monoid.fold_tree(states),
                       monoid.fold_tree([states[j] for j in rng.permutation(len(states))]),
                       monoid.fold_left([monoid.leaf(s[j], V[j]) for j in range(n)])):
                o, lse = monoid.finish(st)
                assert _relerr(o, O[0, h, i]) <= 1e-12, ("regrouped O", h, i)
                assert abs(lse - L[0, h, i]) <= 1e-12 * max(1.0, abs(L[0, h, i])), ("regrouped LSE",)
            # A stale (larger) reference value gives the same O and LSE.
            full = monoid.fold_left(states)
            o, lse = monoid.finish(monoid.with_reference(full, full[0] + 7.5))
            assert _relerr(o, O[0, h, i]) <= 1e-12 and abs(lse - L[0, h, i]) <= 1e-12 * max(1.0, abs(L[0, h, i]))
            # The identity is neutral.
            o1, _ = monoid.finish(full)
            o2, _ = monoid.finish(monoid.combine(monoid.identity(D), full))
            assert _relerr(o2, o1) <= 1e-15


# ---------------------------------------------------------------------------
# 7. Row-sampled variants agree with the whole-tensor definition.
# ---------------------------------------------------------------------------

def check_row_variants(orc):
    rng = _rng(17)
    B, Hq, Hkv, S, D = 2, 6, 3, 40, 8
    scale = 0.45
    q = rng.standard_normal((B, Hq, S, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    dO = rng.standard_normal((B, Hq, S, D))
    for causal in (True, False):
        O, L = orc.forward(q, k, v, causal=causal, scale=scale, row_block=7)
        dQ, dK, dV = orc.backward(q, k, v, dO, causal=causal, scale=scale)
        rows = np.array([0, 3, 17, 39])
        o, l = orc.forward_rows(q, k, v, 1, 4, rows, causal, scale)
        assert _relerr(o, O[1, 4, rows]) <= 1e-14 and np.max(np.abs(l - L[1, 4, rows])) <= 1e-14
        dq = orc.backward_dq_rows(q, k, v, dO, 1, 5, rows, causal, scale)
        assert _relerr(dq, dQ[1, 5, rows]) <= 1e-12
        dk, dv = orc.backward_dkdv_rows(q, k, v, dO, 0, 2, rows, causal, scale, row_block=9)
        assert _relerr(dk, dK[0, 2, rows]) <= 1e-12 and _relerr(dv, dV[0, 2, rows]) <= 1e-12


# ---------------------------------------------------------------------------
# 8. Stored golden file (written by tests/golden/make_golden.py from the
#    oracle alone) still matches, and is itself pinned by the decimal brute
#    force on its forward.
# ---------------------------------------------------------------------------

def load_golden():
    path = GOLDEN / "small_case.json"
    data = json.loads(path.read_text())
    arr = {k: np.array(v, dtype=np.float64) for k, v in data["arrays"].items()}
    return data["meta"], arr


def check_golden(orc):
    meta, a = load_golden()
    O, L = orc.forward(a["q"], a["k"], a["v"], causal=meta["causal"], scale=meta["scale"])
    dQ, dK, dV = orc.backward(a["q"], a["k"], a["v"], a["dO"], causal=meta["causal"], scale=meta["scale"])
    for name, x in (("O", O), ("LSE", L), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        assert _relerr(x, a[name]) <= 1e-13, ("golden", name, _relerr(x, a[name]))


# ---------------------------------------------------------------------------
# 9. Cached (decode) attention: bottom-right alignment, against the full
#    sequence, a decimal brute force with explicit positions, and torch SDPA
#    with an explicit mask.
# ---------------------------------------------------------------------------

def brute_cached_decimal(q, k, v, causal, scale, prec=50):
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Sq, D))
    L = np.zeros((B, Hq, Sq))
    with localcontext() as ctx:
        ctx.prec = prec
        sc = Decimal(float(scale))
        for b in range(B):
            for h in range(Hq):
                for i in range(Sq):
                    pos = Sk - Sq + i  # absolute position of new query i
                    w = []
                    for j in range(Sk):
                        if causal and j > pos:
                            continue
                        dot = sum(Decimal(float(q[b, h, i, d])) * Decimal(float(k[b, h // G, j, d])) for d in range(D))
                        w.append((j, (sc * dot).exp()))
                    Z = sum(x for _, x in w)
                    for d in range(D):
                        O[b, h, i, d] = float(sum(x * Decimal(float(v[b, h // G, j, d])) for j, x in w) / Z)
                    L[b, h, i] = float(Z.ln())
    return O, L


def check_decode(orc):
    rng = _rng(18)
    # decimal brute force, tiny
    for (B, Hq, Hkv, Sq, Sk, D, causal) in [(1, 4, 2, 2, 5, 3, True), (1, 2, 1, 3, 3, 2, True), (1, 2, 2, 1, 4, 3, False)]:
        q = _dyadic(rng, (B, Hq, Sq, D))
        k = _dyadic(rng, (B, Hkv, Sk, D))
        v = _dyadic(rng, (B, Hkv, Sk, D))
        O, L = orc.forward_cached(q, k, v, causal=causal, scale=0.6)
        Ob, Lb = brute_cached_decimal(q, k, v, causal, 0.6)
        assert _relerr(O, Ob) <= 1e-14 and np.max(np.abs(L - Lb)) <= 1e-13, "cached vs decimal"
    # the last Sq rows of the full-sequence forward
    B, Hq, Hkv, Sk, Sq, D = 2, 6, 2, 33, 5, 8
    qf = rng.standard_normal((B, Hq, Sk, D))
    k = rng.standard_normal((B, Hkv, Sk, D))
    v = rng.standard_normal((B, Hkv, Sk, D))
    for causal in (True, False):
        Of, Lf = orc.forward(qf, k, v, causal=causal, scale=0.4)
        O, L = orc.forward_cached(qf[:, :, -Sq:], k, v, causal=causal, scale=0.4)
        assert _relerr(O, Of[:, :, -Sq:]) <= 1e-14 and np.max(np.abs(L - Lf[:, :, -Sq:])) <= 1e-14, "cached = tail"
    # torch f64 SDPA with an explicit bottom-right mask
    q = rng.standard_normal((B, Hq, Sq, D))
    G = Hq // Hkv
    mask = torch.arange(Sk)[None, :] <= (Sk - Sq + torch.arange(Sq))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k).repeat_interleave(G, dim=1), torch.tensor(v).repeat_interleave(G, dim=1),
        attn_mask=mask, scale=0.4)
    O, _ = orc.forward_cached(q, k, v, causal=True, scale=0.4)
    assert _relerr(O, ref.numpy()) <= 1e-12, "cached vs torch SDPA"


# ---------------------------------------------------------------------------
# 10. Packed variable-length batches: torch f64 SDPA over the whole pack with an
#     explicit mask (same sequence, bottom-right causal within it), forward and
#     autograd backward; reversing the order of the sequences in the pack
#     reverses the result.
# ---------------------------------------------------------------------------

def _pack_mask(cq, ck, causal):
    Tq, Tk = int(cq[-1]), int(ck[-1])
    mask = torch.zeros(Tq, Tk, dtype=torch.bool)
    for i in range(len(cq) - 1):
        nq, nk = int(cq[i + 1] - cq[i]), int(ck[i + 1] - ck[i])
        r = torch.arange(nq)[:, None]
        j = torch.arange(nk)[None, :]
        blk = (j <= (nk - nq) + r) if causal else torch.ones(nq, nk, dtype=torch.bool)
        mask[cq[i]:cq[i + 1], ck[i]:ck[i + 1]] = blk
    return mask


def _sdpa_pack(q, k, v, cq, ck, causal, scale, G):
    mask = _pack_mask(cq, ck, causal)
    return torch.nn.functional.scaled_dot_product_attention(
        q[None], k.repeat_interleave(G, dim=0)[None], v.repeat_interleave(G, dim=0)[None],
        attn_mask=mask, scale=scale)[0]


def check_varlen(orc):
    rng = _rng(19)
    Hq, Hkv, D, scale = 6, 2, 8, 0.45
    G = Hq // Hkv
    # forward: separate query and key bounds, an empty sequence, Sq < Sk and Sq = Sk
    cq = np.array([0, 3, 3, 10, 11])
    ck = np.array([0, 5, 7, 14, 19])
    q = rng.standard_normal((Hq, cq[-1], D))
    k = rng.standard_normal((Hkv, ck[-1], D))
    v = rng.standard_normal((Hkv, ck[-1], D))
    for causal in (True, False):
        O, L = orc.forward_varlen(q, k, v, cq, ck, causal=causal, scale=scale)
        ref = _sdpa_pack(torch.tensor(q), torch.tensor(k), torch.tensor(v), cq, ck, causal, scale, G)
        assert _relerr(O, ref.numpy()) <= 1e-12, f"varlen forward vs torch SDPA (causal={causal})"
        s = scale * np.einsum("htd,hsd->hts", q, np.repeat(k, G, axis=0))
        s = np.where(_pack_mask(cq, ck, causal).numpy()[None], s, -np.inf)
        m = s.max(axis=2)
        assert np.max(np.abs(L - (m + np.log(np.exp(s - m[..., None]).sum(axis=2))))) <= 1e-12, "varlen LSE"
    # backward, packed self-attention
    cu = np.array([0, 4, 5, 12, 12, 20])
    T = int(cu[-1])
    q = rng.standard_normal((Hq, T, D))
    k = rng.standard_normal((Hkv, T, D))
    v = rng.standard_normal((Hkv, T, D))
    dO = rng.standard_normal((Hq, T, D))
    for causal in (True, False):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        out = _sdpa_pack(tq, tk, tv, cu, cu, causal, scale, G)
        (out * torch.tensor(dO)).sum().backward()
        dQ, dK, dV = orc.backward_varlen(q, k, v, dO, cu, causal=causal, scale=scale)
        for name, mine, ref in (("dQ", dQ, tq.grad), ("dK", dK, tk.grad), ("dV", dV, tv.grad)):
            assert _relerr(mine, ref.numpy()) <= 1e-11, f"varlen {name} vs torch autograd (causal={causal})"
    # reversing the sequences of the pack reverses the result
    lens = np.diff(cu)
    rev_cu = np.concatenate([[0], np.cumsum(lens[::-1])])
    perm = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in reversed(range(len(lens)))])
    O1, L1 = orc.forward_varlen(q, k, v, cu, cu, causal=True, scale=scale)
    O2, L2 = orc.forward_varlen(q[:, perm], k[:, perm], v[:, perm], rev_cu, rev_cu, causal=True, scale=scale)
    assert np.array_equal(O1[:, perm], O2) and np.array_equal(L1[:, perm], L2), "varlen pack order"


# ---------------------------------------------------------------------------
# 11. Rotary position embedding: the rotation against complex multiplication,
#     norms kept, scores that depend only on the distance between positions,
#     central finite differences of L = sum(O * dO) through the rotation, and
#     torch f64 autograd of an explicit rotation followed by SDPA.
# ---------------------------------------------------------------------------

def _tables64(S, D, base=10000.0, offset=0):
    i = np.arange(D // 2)
    ang = (offset + np.arange(S))[:, None] * base ** (-2.0 * i / D)[None, :]
    return np.cos(ang), np.sin(ang)


def check_rope(orc):
    rng = _rng(20)
    S, D = 9, 8
    cos, sin = _tables64(S, D)
    x = rng.standard_normal((2, 3, S, D))
    xr = orc.rope.rotate(x, cos, sin)
    z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * np.arctan2(sin, cos))
    assert _relerr(xr, np.concatenate([z.real, z.imag], axis=-1)) <= 1e-14, "rotation vs complex product"
    assert np.max(np.abs(np.linalg.norm(xr, axis=-1) - np.linalg.norm(x, axis=-1))) <= 1e-13, "norm kept"
    assert _relerr(orc.rope.unrotate(xr, cos, sin), x) <= 1e-14, "unrotate inverts rotate"
    # scores depend on positions only through their difference
    q = rng.standard_normal((S, D))
    k = rng.standard_normal((S, D))
    c2, s2 = _tables64(S, D, offset=37)
    s_a = orc.rope.rotate(q, cos, sin) @ orc.rope.rotate(k, cos, sin).T
    s_b = orc.rope.rotate(q, c2, s2) @ orc.rope.rotate(k, c2, s2).T
    assert np.max(np.abs(s_a - s_b)) <= 1e-12, "relative-position property"
    # gradients through the rotation: central finite differences
    B, Hq, Hkv, S, D = 1, 4, 2, 6, 4
    cos, sin = _tables64(S, D, base=3.0)
    q = rng.standard_normal((B, Hq, S, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    dO = rng.standard_normal((B, Hq, S, D))
    dQ, dK, dV = orc.backward_rope(q, k, v, dO, cos, sin, causal=True, scale=0.7)

    def loss(qq, kk, vv):
        return float(np.sum(orc.forward_rope(qq, kk, vv, cos, sin, causal=True, scale=0.7)[0] * dO))

    h = 1e-5
    for name, X, G in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp = X.copy()
            Xm = X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"q": (Xp, k, v), "k": (q, Xp, v), "v": (q, k, Xp)}[name]
            args_m = {"q": (Xm, k, v), "k": (q, Xm, v), "v": (q, k, Xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert _relerr(G, num) <= 1e-6, f"rope d{name} vs finite differences"
    # torch f64: explicit rotation, SDPA, autograd
    G_ = Hq // Hkv
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (q, k, v))
    tc, ts = torch.tensor(cos), torch.tensor(sin)

    def trot(t):
        lo, hi = t[..., : D // 2], t[..., D // 2:]
        return torch.cat([lo * tc - hi * ts, hi * tc + lo * ts], dim=-1)

    out = torch.nn.functional.scaled_dot_product_attention(
        trot(tq), trot(tk).repeat_interleave(G_, dim=1), tv.repeat_interleave(G_, dim=1), is_causal=True, scale=0.7)
    (out * torch.tensor(dO)).sum().backward()
    O, _ = orc.forward_rope(q, k, v, cos, sin, causal=True, scale=0.7)
    assert _relerr(O, out.detach().numpy()) <= 1e-12, "rope forward vs torch"
    for name, mine, ref in (("dQ", dQ, tq.grad), ("dK", dK, tk.grad), ("dV", dV, tv.grad)):
        assert _relerr(mine, ref.numpy()) <= 1e-11, f"rope {name} vs torch autograd"


ALL_CHECKS = [
    "check_decimal_bruteforce",
    "check_finite_differences",
    "check_closed_forms",
    "check_invariants",
    "check_torch_sdpa",
    "check_monoid_regrouping",
    "check_row_variants",
    "check_golden",
    "check_decode",
    "check_varlen",
    "check_rope",
]
