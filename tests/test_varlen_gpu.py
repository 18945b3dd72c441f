"""GPU parity of packed variable-length batches (sequences laid end to end along the token axis)
with the f64 oracle's ``forward_varlen`` and ``backward_varlen``."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_fwd_close, assert_grad_close, gqa
from gqa_inputs import draw_lengths, make_inputs, make_packed_inputs, to_f64

pytestmark = pytest.mark.gpu


def _fwd_case(g, Hq, Hkv, lens_q, lens_k, D, seed, causal=True):
    q, k, v, _, cu_q, cu_k = make_packed_inputs(Hq, Hkv, lens_q, lens_k, D, seed, with_do=False)
    scale = 1.0 / np.sqrt(D)
    o, lse = g.gqa_attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lens_q),
                                   causal=causal, scale=scale)
    assert g.gqa_attn_get_error() == 0
    O_ref, L_ref = oracle.forward_varlen(to_f64(q), to_f64(k), to_f64(v), cu_q.numpy(), cu_k.numpy(),
                                         causal=causal, scale=scale)
    # the [H, T, D] pack read as a batch of one
    assert_fwd_close(o.float().cpu().numpy()[None], lse.cpu().numpy()[None], O_ref[None], L_ref[None],
                     f"varlen Hq={Hq} Hkv={Hkv} lens_q={lens_q} lens_k={lens_k} D={D} causal={causal}")


# Lengths around the 128-row tile and the 256-row CTA pair, an empty sequence, one-row sequences.
PACKS = [
    [1],
    [300],
    [1, 127, 128, 129],
    [255, 0, 256, 257, 3],
    [513, 64, 1, 200],
]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lens", PACKS)
def test_packed_self_attention(lens, D):
    g = gqa()
    _fwd_case(g, 4, 2, lens, lens, D, seed=sum(lens) + D)


@pytest.mark.parametrize("lens", [[130, 5, 400], [1, 1, 1]])
def test_packed_non_causal(lens):
    g = gqa()
    _fwd_case(g, 6, 3, lens, lens, 64, seed=7 + len(lens), causal=False)


def test_packed_queries_over_caches():
    """Each sequence: a few new queries over its own longer cache (bottom-right causal)."""
    g = gqa()
    _fwd_case(g, 8, 2, [1, 100, 129, 0, 260], [300, 100, 700, 5, 261], 128, seed=3)


def test_packed_many_random_lengths():
    g = gqa()
    lens = draw_lengths(24, 1, 700, seed=12)
    _fwd_case(g, 8, 8, lens, lens, 128, seed=12)


def test_equal_lengths_equal_dense_batch():
    """A pack of B sequences of one length equals the dense [B, H, S, D] forward bitwise."""
    g = gqa()
    B, Hq, Hkv, S, D = 3, 8, 2, 333, 128
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_inputs(B, Hq, Hkv, S, D, 17, with_do=False))
    o_d, l_d = g.gqa_attn_fwd(q, k, v)

    def pack(x):  # [B, H, S, D] -> [H, B*S, D]
        return x.permute(1, 0, 2, 3).reshape(x.shape[1], B * S, D).contiguous()

    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    o_p, l_p = g.gqa_attn_fwd_varlen(pack(q), pack(k), pack(v), cu, cu, S)
    assert torch.equal(o_p, pack(o_d))
    assert torch.equal(l_p, l_d.permute(1, 0, 2).reshape(Hq, B * S))


def test_invalid_device_bounds_are_reported():
    """Bounds live on the device: invalid ones are skipped by the kernel and reported afterwards,
    while the valid sequences of the same call are computed."""
    g = gqa()
    Hq, Hkv, D, T = 4, 2, 64, 300
    q, k, v, _, _, _ = make_packed_inputs(Hq, Hkv, [T], [T], D, seed=5, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    cases = [
        [0, 100, 50, 300],    # decreasing
        [0, 100, 400, 300],   # past the end of the rows
        [0, 299, 300, 300],   # a 299-row sequence with max_seqlen_q = 200
    ]
    for cu in cases:
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        o = torch.zeros_like(q)
        lse = torch.zeros(Hq, T, device="cuda")
        g.gqa_attn_fwd_varlen(q, k, v, cu_d, cu_d, 200, o=o, lse=lse)
        assert g.gqa_attn_get_error() == g.GQA_ERR_INVALID_ARG, cu
    # more queries than keys in one sequence
    cu_q = torch.tensor([0, 10, 300], dtype=torch.int32, device="cuda")
    cu_k = torch.tensor([0, 5, 300], dtype=torch.int32, device="cuda")
    o, lse = g.gqa_attn_fwd_varlen(q, k, v, cu_q, cu_k, 290)
    assert g.gqa_attn_get_error() == g.GQA_ERR_INVALID_ARG
    # the valid second sequence was still computed
    O_ref, L_ref = oracle.forward_cached(to_f64(q[None, :, 10:]), to_f64(k[None, :, 5:]), to_f64(v[None, :, 5:]))
    assert_fwd_close(o[None, :, 10:].float().cpu().numpy(), lse[None, :, 10:].cpu().numpy(), O_ref, L_ref,
                     "valid sequence next to an invalid one")
    assert g.gqa_attn_get_error() == 0


def test_host_rejects_bad_arguments():
    g = gqa()
    q = torch.zeros(4, 64, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(2, 64, 64, device="cuda", dtype=torch.bfloat16)
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    with pytest.raises(g.GqaAttnError):
        g.gqa_attn_fwd_varlen(q, k, k, cu, cu, 65)  # max_seqlen_q > Tq
    with pytest.raises(g.GqaAttnError):
        g.gqa_attn_fwd_varlen(q, k, k, cu, cu, 0)
    with pytest.raises(ValueError):
        g.gqa_attn_fwd_varlen(q, k, k, cu.long(), cu, 64)


def _fwd_bwd_case(g, Hq, Hkv, lens, D, seed, causal=True):
    """Packed self-attention: forward, then backward from the forward's O and LSE."""
    q, k, v, dO, cu, _ = make_packed_inputs(Hq, Hkv, lens, lens, D, seed)
    scale = 1.0 / np.sqrt(D)
    qd, kd, vd, dOd, cud = q.cuda(), k.cuda(), v.cuda(), dO.cuda(), cu.cuda()
    o, lse = g.gqa_attn_fwd_varlen(qd, kd, vd, cud, cud, max(lens), causal=causal, scale=scale)
    dq, dk, dv = g.gqa_attn_bwd_varlen(qd, kd, vd, o, dOd, lse, cud, max(lens), causal=causal, scale=scale)
    assert g.gqa_attn_get_error() == 0
    qf, kf, vf, dOf = (to_f64(t) for t in (q, k, v, dO))
    where = f"varlen bwd Hq={Hq} Hkv={Hkv} lens={lens} D={D} causal={causal}"
    O_ref, L_ref = oracle.forward_varlen(qf, kf, vf, cu.numpy(), cu.numpy(), causal=causal, scale=scale)
    assert_fwd_close(o.float().cpu().numpy()[None], lse.cpu().numpy()[None], O_ref[None], L_ref[None], where)
    dQ, dK, dV = oracle.backward_varlen(qf, kf, vf, dOf, cu.numpy(), causal=causal, scale=scale)
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        assert_grad_close(name, got.float().cpu().numpy(), ref, where)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lens", PACKS)
def test_packed_backward(lens, D):
    g = gqa()
    _fwd_bwd_case(g, 4, 2, lens, D, seed=sum(lens) * 3 + D)


@pytest.mark.parametrize("lens", [[130, 5, 400], [1, 1, 1]])
def test_packed_backward_non_causal(lens):
    g = gqa()
    _fwd_bwd_case(g, 6, 3, lens, 64, seed=11 + len(lens), causal=False)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (12, 4), (16, 1)])
def test_packed_backward_head_groupings(Hq, Hkv):
    g = gqa()
    _fwd_bwd_case(g, Hq, Hkv, [1, 200, 383, 4, 129], 128, seed=Hq + Hkv)


def test_packed_backward_many_random_lengths():
    g = gqa()
    lens = draw_lengths(20, 1, 600, seed=13)
    _fwd_bwd_case(g, 8, 2, lens, 128, seed=13)


def test_packed_backward_equals_dense_batch():
    """At equal lengths the packed backward matches the dense one within f32 summation-order noise
    (the dense backward of a problem this small splits its key tiles over several CTAs and adds
    their partials; the packed one sums each key tile in one CTA)."""
    g = gqa()
    B, Hq, Hkv, S, D = 3, 8, 2, 333, 128
    q, k, v, dO = (t.cuda() for t in make_inputs(B, Hq, Hkv, S, D, 19))
    o, lse = g.gqa_attn_fwd(q, k, v)
    dq_d, dk_d, dv_d = g.gqa_attn_bwd(q, k, v, o, dO, lse)

    def pack(x):  # [B, H, S, D] -> [H, B*S, D]
        return x.permute(1, 0, 2, 3).reshape(x.shape[1], B * S, x.shape[3]).contiguous()

    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    lse_p = lse.permute(1, 0, 2).reshape(Hq, B * S).contiguous()
    dq_p, dk_p, dv_p = g.gqa_attn_bwd_varlen(pack(q), pack(k), pack(v), pack(o), pack(dO), lse_p, cu, S)
    assert g.gqa_attn_get_error() == 0
    for got, want in ((dk_p, pack(dk_d)), (dv_p, pack(dv_d)), (dq_p, pack(dq_d))):
        assert (got.float() - want.float()).abs().max().item() <= 1e-2 * want.float().abs().max().item()


def test_packed_backward_invalid_bounds_reported():
    g = gqa()
    Hq, Hkv, D, T = 4, 2, 64, 300
    q, k, v, dO, _, _ = make_packed_inputs(Hq, Hkv, [T], [T], D, seed=6)
    q, k, v, dO = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o = torch.zeros_like(q)
    lse = torch.zeros(Hq, T, device="cuda")
    for cu, max_len in (([0, 100, 50, 300], 300), ([0, 100, 400, 300], 300), ([0, 299, 300, 300], 200)):
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        g.gqa_attn_bwd_varlen(q, k, v, o, dO, lse, cu_d, max_len)
        assert g.gqa_attn_get_error() == g.GQA_ERR_INVALID_ARG, cu
