"""GPU parity of attention with the rotary position embedding fused in (rotate-half pairing,
caller tables) against the f64 oracle's ``forward_rope`` / ``backward_rope``.

The kernels feed the tensor cores bf16 operands, so the rotated q and k are rounded to bf16
(as any bf16 attention over rotated inputs must). Two comparisons:
* forward against the oracle's plain attention over the bf16-rounded rotated operands
  (rounded here, in f32, from the same tables), at the standard tolerances;
* gradients against the exact f64 ``backward_rope`` at the standard gradient tolerance, and
  the forward against the exact ``forward_rope`` within the bound the bf16 rounding of the
  rotated operands implies: each score moves by at most scale * 2^-8 * |q'_i| * max_j |k'_j|
  (two roundings of 2^-9 relative, Cauchy-Schwarz), so LSE by at most that much.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL_LSE, assert_fwd_close, assert_grad_close, gqa
from gqa_inputs import make_inputs, rope_tables, to_f64

pytestmark = pytest.mark.gpu


def _rotate_bf16(x, cos, sin):
    """bf16(rotate(x)) computed in f32 on the CPU: the operand the tensor cores see."""
    h = x.shape[-1] // 2
    xf = x.float()
    lo, hi = xf[..., :h], xf[..., h:]
    return torch.cat([lo * cos - hi * sin, hi * cos + lo * sin], dim=-1).to(torch.bfloat16)


def _case(g, B, Hq, Hkv, S, D, seed, causal=True, base=10000.0, with_bwd=True):
    q, k, v, dO = make_inputs(B, Hq, Hkv, S, D, seed)
    cos, sin = rope_tables(S, D, base)
    scale = 1.0 / np.sqrt(D)
    qd, kd, vd, dOd, cd, sd = (t.cuda() for t in (q, k, v, dO, cos, sin))
    o, lse = g.gqa_attn_fwd_rope(qd, kd, vd, cd, sd, causal=causal, scale=scale)
    assert g.gqa_attn_get_error() == 0
    where = f"rope (B={B},Hq={Hq},Hkv={Hkv},S={S},D={D},causal={causal},base={base:g})"
    O, L = o.float().cpu().numpy(), lse.cpu().numpy()
    # 1. against plain attention over the bf16-rounded rotated operands
    qr, kr = _rotate_bf16(q, cos, sin), _rotate_bf16(k, cos, sin)
    O_r, L_r = oracle.forward(to_f64(qr), to_f64(kr), to_f64(v), causal=causal, scale=scale)
    assert_fwd_close(O, L, O_r, L_r, where + " vs rounded operands")
    # 2. against the exact rotary attention, LSE within the rounding bound
    cf, sf = to_f64(cos), to_f64(sin)
    O_x, L_x = oracle.forward_rope(to_f64(q), to_f64(k), to_f64(v), cf, sf, causal=causal, scale=scale)
    qn = np.linalg.norm(oracle.rope.rotate(to_f64(q), cf, sf), axis=-1)
    kn = np.linalg.norm(oracle.rope.rotate(to_f64(k), cf, sf), axis=-1).max()
    bound = TOL_LSE + scale * 2.0 ** -8 * qn * kn
    assert np.all(np.abs(L - L_x) <= bound), f"{where} LSE beyond the rounding bound"
    assert np.max(np.abs(O - O_x)) <= 5e-2, f"{where} O far from the exact rotary attention"
    if with_bwd:
        dq, dk, dv = g.gqa_attn_bwd_rope(qd, kd, vd, o, dOd, lse, cd, sd, causal=causal, scale=scale)
        assert g.gqa_attn_get_error() == 0
        dQ, dK, dV = oracle.backward_rope(to_f64(q), to_f64(k), to_f64(v), to_f64(dO), cf, sf, causal=causal,
                                          scale=scale)
        for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
            assert_grad_close(name, got.float().cpu().numpy(), ref, where)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 127, 129, 300])
def test_rope_parity(S, D):
    g = gqa()
    _case(g, 1, 4, 2, S, D, seed=S + 3 * D)


@pytest.mark.parametrize("base", [10000.0, 1.0e6])
def test_rope_bases(base):
    g = gqa()
    _case(g, 2, 8, 2, 257, 128, seed=31, base=base)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (12, 4), (16, 1)])
def test_rope_head_groupings(Hq, Hkv):
    g = gqa()
    _case(g, 1, Hq, Hkv, 200, 64, seed=Hq + Hkv)


def test_rope_non_causal():
    g = gqa()
    _case(g, 2, 6, 3, 190, 128, seed=41, causal=False)


def test_identity_tables_equal_plain_attention():
    """cos = 1, sin = 0 turns nothing: outputs equal the plain path bitwise, gradients within f32
    summation-order noise (the plain backward splits the key tiles of a problem this small over
    several CTAs; the rotary one does not)."""
    g = gqa()
    B, Hq, Hkv, S, D = 2, 8, 2, 333, 128
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, S, D, 43))
    cos = torch.ones(S, D // 2, device="cuda")
    sin = torch.zeros(S, D // 2, device="cuda")
    o1, l1 = g.gqa_attn_fwd(q, k, v)
    o2, l2 = g.gqa_attn_fwd_rope(q, k, v, cos, sin)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    dq1, dk1, dv1 = g.gqa_attn_bwd(q, k, v, o1, dO, l1)
    dq2, dk2, dv2 = g.gqa_attn_bwd_rope(q, k, v, o1, dO, l1, cos, sin)
    for a, b in ((dq1, dq2), (dk1, dk2), (dv1, dv2)):
        assert (a.float() - b.float()).abs().max().item() <= 1e-2 * a.float().abs().max().item()


def test_rope_rejects_bad_tables():
    g = gqa()
    q, k, v, _ = (t.cuda() for t in make_inputs(1, 4, 2, 64, 64, 1))
    cos = torch.ones(63, 32, device="cuda")
    with pytest.raises(ValueError):
        g.gqa_attn_fwd_rope(q, k, v, cos, cos)
