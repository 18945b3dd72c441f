"""Shared helpers of the GPU tests: build/load the library, run it, compare with the oracle."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import make_inputs, to_f64

# Tolerances (stated for this path): O max-abs <= 1e-2, LSE max-abs <= 1e-3,
# dQ/dK/dV max-abs <= 2e-2 * max|ref| per tensor, all against the f64 oracle.
# Gradients that vanish identically (S = 1 gives dQ = dK = 0 exactly) make the
# relative bound empty; there the f32 cancellation of dP - D (two f32 sums of
# D bf16 products, in different orders) leaves ~1e-7, so an absolute floor of
# 1e-5 is added to the gradient bound.
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2
TOL_GRAD_ABS_FLOOR = 1e-5


def gqa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_flash_gb300 import _lib
    from causal_gqa_attention_flash_gb300.build import build_library
    build_library(debug=_lib.DEBUG)  # the variant the binding loads (GQA_ATTN_DEBUG=1: the checking build)
    import causal_gqa_attention_flash_gb300 as g
    return g


def run_gpu(g, q, k, v, dO, causal, scale, with_bwd=True):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = g.gqa_attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    out = {"O": o, "LSE": lse}
    if with_bwd:
        dOd = dO.cuda()
        dq, dk, dv = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, causal=causal, scale=scale)
        out.update(dQ=dq, dK=dk, dV=dv)
    assert g.gqa_attn_get_error() == 0
    return {k_: v_.float().cpu().numpy().astype(np.float64) for k_, v_ in out.items()}


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0


def bf16_half_ulp(x):
    """Half the spacing of bf16 values around |x| (bf16 has an 8-bit significand)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def assert_fwd_close(O, L, O_ref, L_ref, where="", v_absmax=None):
    # O is delivered in bf16, whose half-ulp (0.0156 on [4, 8)) exceeds 1e-2 for |O| >= 4, where no
    # bf16 output can meet 1e-2: there the bound is 1e-2 plus the half-ulp of the exact value.
    O_ref = np.asarray(O_ref, dtype=np.float64)
    bound = TOL_O + np.where(np.abs(O_ref) >= 4.0, bf16_half_ulp(O_ref), 0.0)
    if v_absmax is not None:
        # Peaked rows (scale above 1/sqrt(D)): P enters P.V as bf16 (relative error <= 2^-9 per
        # weight, which no longer averages out when one key dominates), and O is rounded to bf16:
        # |dO| <= 2^-9 (max|v| + |O|), plus 1e-3 for the f32 arithmetic.
        bound = np.maximum(bound, 2.0 ** -9 * (v_absmax + np.abs(O_ref)) + 1e-3)
    excess = float(np.max(np.abs(np.asarray(O) - O_ref) - bound)) if np.size(O) else -1.0
    eo, el = max_abs(O, O_ref), max_abs(L, L_ref)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), where
    assert excess <= 0.0, f"{where} O max-abs err {eo:.3e} exceeds the bound by {excess:.3e}"
    assert el <= TOL_LSE, f"{where} LSE max-abs err {el:.3e} > {TOL_LSE}"


def assert_grad_close(name, X, X_ref, where=""):
    ref_max = float(np.max(np.abs(X_ref))) if np.size(X_ref) else 0.0
    err = max_abs(X, X_ref)
    assert np.all(np.isfinite(X)), f"{where} {name} not finite"
    assert err <= TOL_GRAD_REL * ref_max + TOL_GRAD_ABS_FLOOR, \
        f"{where} {name} max-abs err {err:.3e} > {TOL_GRAD_REL} * {ref_max:.3e}"


def full_case(g, B, Hq, Hkv, S, D, seed, causal=True, do_std=0.1, scale=None, with_bwd=True):
    peaked = scale is not None and scale > 1.0 / np.sqrt(D)
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    q, k, v, dO = make_inputs(B, Hq, Hkv, S, D, seed, do_std=do_std)
    got = run_gpu(g, q, k, v, dO, causal, scale, with_bwd)
    qf, kf, vf, dOf = (to_f64(t) for t in (q, k, v, dO))
    O_ref, L_ref = oracle.forward(qf, kf, vf, causal=causal, scale=scale)
    where = f"(B={B},Hq={Hq},Hkv={Hkv},S={S},D={D},causal={causal},scale={scale:.4g})"
    assert_fwd_close(got["O"], got["LSE"], O_ref, L_ref, where,
                     v_absmax=float(np.max(np.abs(vf))) if peaked else None)
    if with_bwd:
        dQ, dK, dV = oracle.backward(qf, kf, vf, dOf, causal=causal, scale=scale)
        assert_grad_close("dQ", got["dQ"], dQ, where)
        assert_grad_close("dK", got["dK"], dK, where)
        assert_grad_close("dV", got["dV"], dV, where)
    return got
