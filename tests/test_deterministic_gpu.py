"""GPU parity of the deterministic backward (query-major dQ, KV-major dK/dV) with the f64 oracle,
its bitwise reproducibility, and its agreement with the reduce-add backward."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL_GRAD_REL, assert_grad_close, gqa, max_abs
from gqa_inputs import WORKLOADS, make_inputs, to_f64, workload_inputs

pytestmark = pytest.mark.gpu


def _case(g, B, Hq, Hkv, S, D, seed, causal=True, do_std=0.1):
    q, k, v, dO = make_inputs(B, Hq, Hkv, S, D, seed, do_std=do_std)
    scale = 1.0 / np.sqrt(D)
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = g.gqa_attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, causal=causal, scale=scale, deterministic=True)
    assert g.gqa_attn_get_error() == 0
    qf, kf, vf, dOf = (to_f64(t) for t in (q, k, v, dO))
    dQ, dK, dV = oracle.backward(qf, kf, vf, dOf, causal=causal, scale=scale)
    where = f"deterministic (B={B},Hq={Hq},Hkv={Hkv},S={S},D={D},causal={causal})"
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        assert_grad_close(name, got.float().cpu().numpy(), ref, where)


# One row, ragged tails around the 64-key halves and the 128-row tiles, several tiles.
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 63, 64, 65, 127, 128, 129, 200, 385])
def test_deterministic_parity(S, D):
    g = gqa()
    _case(g, 1, 4, 2, S, D, seed=S * 7 + D)


@pytest.mark.parametrize("S", [100, 300])
def test_deterministic_non_causal(S):
    g = gqa()
    _case(g, 2, 6, 3, S, 64, seed=S + 1, causal=False)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (12, 4), (16, 1)])
def test_deterministic_head_groupings(Hq, Hkv):
    g = gqa()
    _case(g, 2, Hq, Hkv, 257, 128, seed=Hq * 3 + Hkv)


@pytest.mark.parametrize("name", ["tiny", "lm101m"])
def test_deterministic_named_workloads(name):
    g = gqa()
    w = WORKLOADS[name]
    _case(g, w.B, w.Hq, w.Hkv, w.S, w.D, w.seed, do_std=w.do_std)


def test_bitwise_reproducible_and_matches_reduce_add_path():
    """Three runs give identical bits; dK and dV equal the reduce-add backward's bitwise (the same
    KV-major element-wise work in the same order), dQ agrees within f32 reduction-order noise."""
    g = gqa()
    q, k, v, dO = (t.cuda() for t in make_inputs(2, 16, 4, 1000, 128, 23))
    o, lse = g.gqa_attn_fwd(q, k, v)
    runs = [g.gqa_attn_bwd(q, k, v, o, dO, lse, deterministic=True) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    dq_a, dk_a, dv_a = g.gqa_attn_bwd(q, k, v, o, dO, lse)
    dq_d, dk_d, dv_d = runs[0]
    assert torch.equal(dk_a, dk_d) and torch.equal(dv_a, dv_d)
    assert (dq_a.float() - dq_d.float()).abs().max().item() <= 1e-2 * dq_a.float().abs().max().item()


def test_deterministic_fullsize_sampled():
    """The Qwen3-8B-style workload (1, 32, 8, 4096, 128) at full size: sampled dQ rows against the
    oracle, and dK/dV equal to the reduce-add backward's bitwise."""
    g = gqa()
    w = WORKLOADS["qwen3_8b"]
    q, k, v, dO = workload_inputs("qwen3_8b")
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = g.gqa_attn_fwd(qd, kd, vd, scale=w.scale)
    dq, dk, dv = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, scale=w.scale, deterministic=True)
    dq_a, dk_a, dv_a = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, scale=w.scale)
    assert g.gqa_attn_get_error() == 0
    assert torch.equal(dk, dk_a) and torch.equal(dv, dv_a)
    dQ = dq.float().cpu().numpy()
    qf, kf, vf, dOf = (to_f64(t) for t in (q, k, v, dO))
    rows = np.array([0, 1, 127, 128, 129, 2047, 4094, 4095])
    for (b, h) in ((0, 0), (0, 31), (0, 17)):
        ref = oracle.backward_dq_rows(qf, kf, vf, dOf, b, h, rows, True, w.scale)
        err = max_abs(dQ[b, h, rows], ref)
        assert err <= TOL_GRAD_REL * np.max(np.abs(dQ[b, h])), f"dQ rows b={b} h={h}: {err:.3e}"
