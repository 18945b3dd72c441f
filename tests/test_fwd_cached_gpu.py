"""GPU parity of the tensor-core forward over a key/value cache (Sq <= Sk, bottom-right causal)
with the f64 oracle's ``forward_cached``."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_fwd_close, gqa
from gqa_inputs import make_inputs, to_f64

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Sq, Sk, D, seed):
    # cache = K/V of a seeded length-Sk sequence; the Sq new queries drawn after it
    _, k, v, _ = make_inputs(B, Hq, Hkv, Sk, D, seed, with_do=False)
    q = make_inputs(B, Hq, Hkv, Sq, D, seed + 1000, with_do=False)[0]
    return q, k, v


def _case(g, B, Hq, Hkv, Sq, Sk, D, seed, causal=True):
    q, k, v = _inputs(B, Hq, Hkv, Sq, Sk, D, seed)
    scale = 1.0 / np.sqrt(D)
    o, lse = g.gqa_attn_fwd_cached(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert g.gqa_attn_get_error() == 0
    O_ref, L_ref = oracle.forward_cached(to_f64(q), to_f64(k), to_f64(v), causal=causal, scale=scale)
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
                     f"fwd_cached B={B} Hq={Hq} Hkv={Hkv} Sq={Sq} Sk={Sk} D={D} causal={causal}")


# Offsets Sk - Sq that are 0, under one tile, exactly one tile and ragged several tiles; Sq spans
# one row, a ragged single tile, an odd number of tiles (a CTA with one live tile) and several.
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sq,Sk", [(1, 1), (1, 300), (5, 133), (100, 164), (128, 256), (129, 300),
                                   (200, 1000), (257, 257), (383, 450), (512, 2100)])
def test_causal_prefill_over_cache(Sq, Sk, D):
    g = gqa()
    _case(g, 1, 4, 2, Sq, Sk, D, seed=Sq * 31 + Sk + D)


@pytest.mark.parametrize("Sq,Sk,D", [(1, 129, 64), (130, 700, 128), (300, 301, 64)])
def test_non_causal_over_cache(Sq, Sk, D):
    g = gqa()
    _case(g, 2, 6, 3, Sq, Sk, D, seed=Sq + Sk, causal=False)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (12, 4), (32, 8), (16, 1)])
def test_head_groupings(Hq, Hkv):
    g = gqa()
    _case(g, 2, Hq, Hkv, 160, 480, 128, seed=Hq * 10 + Hkv)


def test_equal_lengths_is_training_forward():
    """Sq = Sk runs the same kernel as gqa_attn_fwd with offset 0: bitwise equal."""
    g = gqa()
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_inputs(2, 8, 2, 700, 128, 8, with_do=False))
    o1, l1 = g.gqa_attn_fwd(q, k, v)
    o2, l2 = g.gqa_attn_fwd_cached(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_suffix_of_training_forward():
    """The last Sq rows of a length-S forward equal the same queries run over the cache."""
    g = gqa()
    B, Hq, Hkv, S, D, Sq = 1, 8, 2, 1111, 64, 300
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_inputs(B, Hq, Hkv, S, D, 9, with_do=False))
    o_full, l_full = g.gqa_attn_fwd(q, k, v)
    o, l = g.gqa_attn_fwd_cached(q[:, :, -Sq:].contiguous(), k, v)
    assert (o.float() - o_full[:, :, -Sq:].float()).abs().max().item() <= 1e-2
    assert (l - l_full[:, :, -Sq:]).abs().max().item() <= 1e-3


def test_agrees_with_split_kv_decode():
    """For up to 16 rows per KV head both the tensor-core forward and the split-KV decode apply."""
    g = gqa()
    q, k, v = (t.cuda() for t in _inputs(2, 16, 8, 2, 3000, 128, seed=21))
    o1, l1 = g.gqa_attn_fwd_cached(q, k, v)
    o2, l2 = g.gqa_attn_decode_fwd(q, k, v)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_rejects_more_queries_than_keys():
    g = gqa()
    q = torch.zeros(1, 4, 65, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 64, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(g.GqaAttnError):
        g.gqa_attn_fwd_cached(q, k, k)


@pytest.mark.slow
def test_prefill_512_over_16k_sampled_heads():
    """Prefill of 512 new tokens over a 16384-key cache (B=2, Hq=32, Hkv=8, D=128) in one launch;
    three (batch, head) pairs, one per KV group boundary, checked against the oracle in full."""
    g = gqa()
    B, Hq, Hkv, Sq, Sk, D = 2, 32, 8, 512, 16384, 128
    q, k, v = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=77)
    o, lse = g.gqa_attn_fwd_cached(q.cuda(), k.cuda(), v.cuda())
    assert g.gqa_attn_get_error() == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    for b, h in ((0, 0), (1, 13), (1, 31)):
        kh = oracle.kv_head_of(h, Hq, Hkv)
        O_ref, L_ref = oracle.forward_cached(to_f64(q[b:b + 1, h:h + 1]), to_f64(k[b:b + 1, kh:kh + 1]),
                                             to_f64(v[b:b + 1, kh:kh + 1]))
        assert_fwd_close(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], O_ref, L_ref, f"prefill512 b={b} h={h}")


# Sizes whose grid is small enough for the forward to split key ranges: a prefill over a cache,
# short self-attention (parts of one key tile, rows that see no key of a part), ragged lengths, a
# single query tile, GQA groupings, D = 64 and 128.
SPLIT_CASES = [(1, 4, 2, 257, 1000, 64), (2, 4, 4, 130, 900, 128), (1, 8, 2, 512, 4096, 128),
               (1, 2, 2, 700, 700, 128), (2, 4, 2, 513, 2500, 64), (1, 3, 1, 129, 2000, 128)]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D", SPLIT_CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_splitkv_forward(B, Hq, Hkv, Sq, Sk, D, causal):
    """The split-key-range forward against the oracle; these sizes do split (a workspace is needed),
    and the result agrees with the unsplit forward over the cache within f32 rounding."""
    g = gqa()
    assert g.gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, D) > 0
    q, k, v = _inputs(B, Hq, Hkv, Sq, Sk, D, seed=Sq + Sk + D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / np.sqrt(D)
    o, lse = g.gqa_attn_fwd_splitkv(qd, kd, vd, causal=causal, scale=scale)
    assert g.gqa_attn_get_error() == 0
    O_ref, L_ref = oracle.forward_cached(to_f64(q), to_f64(k), to_f64(v), causal=causal, scale=scale)
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
                     f"splitkv B={B} Hq={Hq} Hkv={Hkv} Sq={Sq} Sk={Sk} D={D} causal={causal}")
    o2, l2 = g.gqa_attn_fwd_cached(qd, kd, vd, causal=causal, scale=scale)
    assert (o.float() - o2.float()).abs().max().item() <= 1e-2
    assert (lse - l2).abs().max().item() <= 1e-4


def test_splitkv_reproducible_and_workspace_checked():
    """Two calls give the same bits (the parts merge in part order); a short workspace is refused;
    the split launches the forward and the merge."""
    g = gqa()
    B, Hq, Hkv, Sq, Sk, D = 1, 8, 2, 512, 4096, 128
    q, k, v = (t.cuda() for t in _inputs(B, Hq, Hkv, Sq, Sk, D, seed=5))
    need = g.gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, D)
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    g.gqa_attn_trace_arm()
    r1 = g.gqa_attn_fwd_splitkv(q, k, v, workspace=ws)
    tr = g.gqa_attn_trace_collect()
    assert tr["fwd"][0] == 1 and tr["fwd_combine"][0] == 1
    r2 = g.gqa_attn_fwd_splitkv(q, k, v, workspace=ws)
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
    with pytest.raises(g.GqaAttnError) as ei:
        g.gqa_attn_fwd_splitkv(q, k, v, workspace=ws[:need - 256])
    assert ei.value.code == g.GQA_ERR_WORKSPACE_TOO_SMALL
    assert g.gqa_attn_get_error() == 0


def test_splitkv_without_split_equals_cached_forward():
    """Sizes the plan does not split run the ordinary forward: the same bits, no workspace."""
    g = gqa()
    B, Hq, Hkv, S, D = 2, 32, 8, 2048, 128
    assert g.gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, S, S, D) == 0
    q, k, v = (t.cuda() for t in _inputs(B, Hq, Hkv, S, S, D, seed=9))
    g.gqa_attn_trace_arm()
    o1, l1 = g.gqa_attn_fwd_splitkv(q, k, v)
    assert g.gqa_attn_trace_collect()["fwd_combine"][0] == 0
    o2, l2 = g.gqa_attn_fwd(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
