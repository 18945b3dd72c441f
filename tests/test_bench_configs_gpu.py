"""GPU parity at the launch configurations bench.py times beside the main line, on the bench's own
seeded inputs: split-KV decode (8 sequences, one new token over a 16k cache, split count from the
cost model), prefill of 512 tokens over a 16k cache (B=2, and B=1 with split key ranges), the packed batch of 16 mixed-length
sequences, the rotary-embedding step at long16k and the deterministic backward at long16k.

Where the oracle cannot evaluate every element in seconds it evaluates sampled rows one by one.
Every bound comes from oracle values only (gradient bounds: 2e-2 times the largest |reference|
over the sampled rows, plus the absolute floor).
"""

import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_helpers import TOL_GRAD_ABS_FLOOR, TOL_GRAD_REL, TOL_LSE, assert_fwd_close, gqa, max_abs
from gqa_inputs import (WORKLOADS, draw_lengths, make_inputs, make_packed_inputs, rope_tables, to_f64,
                        workload_inputs)

pytestmark = pytest.mark.gpu


def grad_bound(refs):
    return TOL_GRAD_REL * max(float(np.max(np.abs(r))) for r in refs) + TOL_GRAD_ABS_FLOOR


def test_decode_bench_config_all_rows():
    """bench.DECODE in the launch configuration the bench times (num_splits = 0: the cost model's
    split count); every output row against the oracle."""
    g = gqa()
    c = bench.DECODE
    _, k, v, _ = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sk"], c["D"], c["seed"], with_do=False)
    q = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["D"], c["seed"] + 1, with_do=False)[0]
    o, lse = g.gqa_attn_decode_fwd(q.cuda(), k.cuda(), v.cuda(), num_splits=0)
    assert g.gqa_attn_get_error() == 0
    O_ref, L_ref = oracle.forward_cached(to_f64(q), to_f64(k), to_f64(v), causal=True)
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, "decode bench config")


@pytest.mark.parametrize("name", ["PREFILL", "PREFILL_B1"])
def test_prefill_bench_config_sampled_heads(name):
    """bench.PREFILL (B=2) and bench.PREFILL_B1 (B=1, whose key ranges split): 512 new tokens over
    a 16384-key cache through gqa_attn_fwd_splitkv, as the bench launches it; three (batch, head)
    pairs in full."""
    g = gqa()
    c = getattr(bench, name)
    _, k, v, _ = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sk"], c["D"], c["seed"], with_do=False)
    q = make_inputs(c["B"], c["Hq"], c["Hkv"], c["Sq"], c["D"], c["seed"] + 1, with_do=False)[0]
    o, lse = g.gqa_attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda())
    assert g.gqa_attn_get_error() == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    for b, h in ((0, 0), (c["B"] - 1, 13), (c["B"] - 1, c["Hq"] - 1)):
        kh = oracle.kv_head_of(h, c["Hq"], c["Hkv"])
        O_ref, L_ref = oracle.forward_cached(to_f64(q[b:b + 1, h:h + 1]), to_f64(k[b:b + 1, kh:kh + 1]),
                                             to_f64(v[b:b + 1, kh:kh + 1]))
        assert_fwd_close(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], O_ref, L_ref, f"{name} b={b} h={h}")


def test_packed_bench_batch_sequences():
    """bench.PACKED (16 causal sequences, lengths uniform on [512, 3584], seed 8), forward and
    backward as the bench launches them. The shortest and the longest sequence, for the first and
    the last KV group: every row against the oracle on the sequence cut out of the pack (each
    sequence attends only to itself), gradient bounds from the oracle's values over that block."""
    g = gqa()
    c = bench.PACKED
    lens = draw_lengths(c["n"], c["lo"], c["hi"], c["seed"])
    q, k, v, dO, cu, _ = make_packed_inputs(c["Hq"], c["Hkv"], lens, lens, c["D"], c["seed"])
    qd, kd, vd, dOd, cud = q.cuda(), k.cuda(), v.cuda(), dO.cuda(), cu.cuda()
    m = max(lens)
    o, lse = g.gqa_attn_fwd_varlen(qd, kd, vd, cud, cud, m)
    dq, dk, dv = g.gqa_attn_bwd_varlen(qd, kd, vd, o, dOd, lse, cud, m)
    assert g.gqa_attn_get_error() == 0
    O, L = o.float().cpu().numpy(), lse.cpu().numpy()
    dQ, dK, dV = (t.float().cpu().numpy() for t in (dq, dk, dv))
    G = c["Hq"] // c["Hkv"]
    scale = 1.0 / np.sqrt(c["D"])
    for i in (int(np.argmin(lens)), int(np.argmax(lens))):
        s0, n = int(cu[i]), lens[i]
        for gh in (0, c["Hkv"] - 1):
            hs = slice(gh * G, (gh + 1) * G)
            sl = slice(s0, s0 + n)
            # the sequence's KV group as a 1 x G x 1 causal problem of length n
            qf, kf, vf, dOf = (to_f64(q[None, hs, sl]), to_f64(k[None, gh:gh + 1, sl]), to_f64(v[None, gh:gh + 1, sl]),
                               to_f64(dO[None, hs, sl]))
            where = f"packed seq {i} (n={n}) KV group {gh}"
            O_ref, L_ref = oracle.forward(qf, kf, vf, causal=True, scale=scale)
            assert_fwd_close(O[None, hs, sl], L[None, hs, sl], O_ref, L_ref, where)
            dQ_ref, dK_ref, dV_ref = oracle.backward(qf, kf, vf, dOf, causal=True, scale=scale)
            assert max_abs(dQ[hs, sl], dQ_ref[0]) <= grad_bound([dQ_ref]), where + " dQ"
            assert max_abs(dK[gh, sl], dK_ref[0, 0]) <= grad_bound([dK_ref]), where + " dK"
            assert max_abs(dV[gh, sl], dV_ref[0, 0]) <= grad_bound([dV_ref]), where + " dV"


def _rotate_rows_bf16(x, cos, sin):
    """bf16(rotate(x)) in f32 on the CPU (x [..., n, D], tables [n, D/2]): the operand the tensor
    cores see."""
    h = x.shape[-1] // 2
    xf = x.float()
    lo, hi = xf[..., :h], xf[..., h:]
    return torch.cat([lo * cos - hi * sin, hi * cos + lo * sin], dim=-1).to(torch.bfloat16)


def test_rope_long16k_sampled():
    """The bench's rotary step (long16k, tables for base 10000) at full size. Forward rows against
    plain attention over the bf16-rounded rotated operands at the standard tolerances, and LSE
    against the exact rotary attention within the bound the operand rounding implies; gradient
    rows against the exact f64 rotary backward at the standard gradient tolerance."""
    g = gqa()
    w = WORKLOADS["long16k"]
    q, k, v, dO = workload_inputs("long16k")
    cos, sin = rope_tables(w.S, w.D)
    qd, kd, vd, dOd, cd, sd = (t.cuda() for t in (q, k, v, dO, cos, sin))
    o, lse = g.gqa_attn_fwd_rope(qd, kd, vd, cd, sd, scale=w.scale)
    dq, dk, dv = g.gqa_attn_bwd_rope(qd, kd, vd, o, dOd, lse, cd, sd, scale=w.scale)
    assert g.gqa_attn_get_error() == 0
    O, L = o.float().cpu().numpy(), lse.cpu().numpy()
    dQ, dK, dV = (t.float().cpu().numpy() for t in (dq, dk, dv))
    cf, sf = to_f64(cos), to_f64(sin)
    G = w.G
    rows = np.array([0, 1, 127, 128, 129, w.S // 2, w.S - 129, w.S - 1])
    key_rows = np.array([(3 * w.S) // 4, w.S - 300, w.S - 129, w.S - 1])
    for (b, h) in ((0, 0), (w.B - 1, w.Hq - 1)):
        gh = h // G
        hs = slice(gh * G, (gh + 1) * G)
        hl = h - gh * G
        where = f"rope long16k b={b} h={h}"
        # 1. forward against plain attention over the bf16-rounded rotated operands
        qr = _rotate_rows_bf16(q[b:b + 1, hs], cos, sin)
        kr = _rotate_rows_bf16(k[b:b + 1, gh:gh + 1], cos, sin)
        vf = to_f64(v[b:b + 1, gh:gh + 1])
        O_r, L_r = oracle.forward_rows(to_f64(qr), to_f64(kr), vf, 0, hl, rows, True, w.scale)
        assert_fwd_close(O[b, h, rows], L[b, h, rows], O_r, L_r, where + " vs rounded operands")
        # 2. exact rotary attention (f64 rotation of the bf16 inputs)
        qx = oracle.rope.rotate(to_f64(q[b:b + 1, hs]), cf, sf)
        kx = oracle.rope.rotate(to_f64(k[b:b + 1, gh:gh + 1]), cf, sf)
        dOf = to_f64(dO[b:b + 1, hs])
        _, L_x = oracle.forward_rows(qx, kx, vf, 0, hl, rows, True, w.scale)
        bound = TOL_LSE + w.scale * 2.0 ** -8 * np.linalg.norm(qx[0, hl, rows], axis=-1) * \
            np.linalg.norm(kx[0, 0], axis=-1).max()
        assert np.all(np.abs(L[b, h, rows] - L_x) <= bound), where + " LSE beyond the rounding bound"
        gq = oracle.backward_dq_rows(qx, kx, vf, dOf, 0, hl, rows, True, w.scale)
        dQ_ref = oracle.rope.unrotate(gq, cf[rows], sf[rows])
        assert max_abs(dQ[b, h, rows], dQ_ref) <= grad_bound([dQ_ref]), where + " dQ"
        gk, gv = oracle.backward_dkdv_rows(qx, kx, vf, dOf, 0, 0, key_rows, True, w.scale)
        dK_ref = oracle.rope.unrotate(gk, cf[key_rows], sf[key_rows])
        assert max_abs(dK[b, gh, key_rows], dK_ref) <= grad_bound([dK_ref]), where + " dK"
        assert max_abs(dV[b, gh, key_rows], gv) <= grad_bound([gv]), where + " dV"


def test_deterministic_long16k_sampled():
    """The bench's deterministic backward at long16k: dQ rows against the oracle, dK/dV rows
    against the oracle and bitwise equal to the reduce-add backward's (same kernel code and order)."""
    g = gqa()
    w = WORKLOADS["long16k"]
    q, k, v, dO = workload_inputs("long16k")
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = g.gqa_attn_fwd(qd, kd, vd, scale=w.scale)
    dq, dk, dv = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, scale=w.scale, deterministic=True)
    _, dk_a, dv_a = g.gqa_attn_bwd(qd, kd, vd, o, dOd, lse, scale=w.scale)
    assert g.gqa_attn_get_error() == 0
    assert torch.equal(dk, dk_a) and torch.equal(dv, dv_a)
    dQ, dK, dV = (t.float().cpu().numpy() for t in (dq, dk, dv))
    G = w.G
    rows = np.array([0, 1, 127, 128, 129, 8191, 16254, 16383])
    key_rows = np.array([(3 * w.S) // 4, w.S - 300, w.S - 129, w.S - 1])
    for (b, h) in ((0, 0), (1, 31), (0, 17)):
        gh = h // G
        hs = slice(gh * G, (gh + 1) * G)
        qf, kf, vf, dOf = (to_f64(q[b:b + 1, hs]), to_f64(k[b:b + 1, gh:gh + 1]), to_f64(v[b:b + 1, gh:gh + 1]),
                           to_f64(dO[b:b + 1, hs]))
        ref = oracle.backward_dq_rows(qf, kf, vf, dOf, 0, h - gh * G, rows, True, w.scale)
        assert max_abs(dQ[b, h, rows], ref) <= grad_bound([ref]), f"dQ rows b={b} h={h}"
        if h % G == 0:
            dK_ref, dV_ref = oracle.backward_dkdv_rows(qf, kf, vf, dOf, 0, 0, key_rows, True, w.scale)
            assert max_abs(dK[b, gh, key_rows], dK_ref) <= grad_bound([dK_ref]), f"dK rows b={b} g={gh}"
            assert max_abs(dV[b, gh, key_rows], dV_ref) <= grad_bound([dV_ref]), f"dV rows b={b} g={gh}"
