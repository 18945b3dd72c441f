"""Why the backward keeps f32 accumulators: an ablation on the CPU (no GPU).

The page "A compiler that derives GPU kernels matches hand-tuned code"
(aiinsiders.net, the paragraph on the derived kernels' weak spots) reports that
a fused attention backward that computes in bf16 misses the f32 accuracy
tolerance. This test plays a tiled backward both ways on the CPU: the same
exact P and dS, the same tile-by-tile sums of dQ, dK and dV, with the running
accumulator rounded after every 16-deep step (one MMA's depth along the
reduction) either to bf16 or to f32. Against the f64 oracle, under the
gradient gate the GPU parity tests use (max-abs error <= 2e-2 * max|ref| per
tensor), the f32 variant passes and the bf16 one fails: the gate is tight
enough to reject the failure the page describes, and the kernels' f32 TMEM
accumulators are what keeps them inside it.
"""

import numpy as np
import pytest
import torch

import oracle
from gqa_inputs import make_inputs, to_f64

TOL_GRAD_REL = 2e-2  # the gradient gate of the GPU parity tests
STEP = 16            # reduction depth of one bf16 MMA


def _round(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).double().numpy()


def _tiled_backward(q, k, v, dO, scale, acc_dtype):
    """dQ, dK, dV of causal GQA from exact f64 P and dS, summed STEP rows at a time with the
    accumulator rounded to acc_dtype after every step."""
    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    visible = np.tril(np.ones((S, S), dtype=bool))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = np.where(visible, scale * q[b, h] @ k[b, g].T, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[b, g]
            dS = p * (dO[b, h] @ v[b, g].T - (dO[b, h] * o).sum(axis=1, keepdims=True))
            for i0 in range(0, S, STEP):  # key-major sums over query rows
                rows = slice(i0, i0 + STEP)
                dV[b, g] = _round(dV[b, g] + p[rows].T @ dO[b, h, rows], acc_dtype)
                dK[b, g] = _round(dK[b, g] + scale * dS[rows].T @ q[b, h, rows], acc_dtype)
            for j0 in range(0, S, STEP):  # query-major sums over keys
                cols = slice(j0, j0 + STEP)
                dQ[b, h] = _round(dQ[b, h] + scale * dS[:, cols] @ k[b, g, cols], acc_dtype)
    return dQ, dK, dV


def _rel_errors(got, ref):
    return [np.abs(a - r).max() / np.abs(r).max() for a, r in zip(got, ref)]


@pytest.fixture(scope="module")
def case():
    B, Hq, Hkv, S, D = 1, 4, 1, 1024, 64
    q, k, v, dO = (to_f64(t) for t in make_inputs(B, Hq, Hkv, S, D, 5, do_std=0.1))
    scale = 1.0 / np.sqrt(D)
    return q, k, v, dO, scale, oracle.backward(q, k, v, dO, causal=True, scale=scale)


def test_f32_accumulators_pass_the_gate(case):
    q, k, v, dO, scale, ref = case
    errs = _rel_errors(_tiled_backward(q, k, v, dO, scale, torch.float32), ref)
    assert max(errs) <= 1e-5, errs  # f32 rounding of the running sums alone: far inside 2e-2


def test_bf16_accumulators_fail_the_gate(case):
    q, k, v, dO, scale, ref = case
    errs = _rel_errors(_tiled_backward(q, k, v, dO, scale, torch.bfloat16), ref)
    assert max(errs) > TOL_GRAD_REL, errs
