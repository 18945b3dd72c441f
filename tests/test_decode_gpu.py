"""GPU parity of the split-KV decode path (new queries against a KV cache) with the f64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_fwd_close, gqa
from gqa_inputs import make_inputs, to_f64

pytestmark = pytest.mark.gpu


def _case(g, B, Hq, Hkv, Sq, Sk, D, seed, causal=True, num_splits=0):
    # cache = K/V of a seeded length-Sk sequence; new queries drawn after it
    _, k, v, _ = make_inputs(B, Hq, Hkv, Sk, D, seed, with_do=False)
    q = make_inputs(B, Hq, Hkv, Sq, D, seed + 1000, with_do=False)[0]
    scale = 1.0 / np.sqrt(D)
    o, lse = g.gqa_attn_decode_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, num_splits=num_splits)
    assert g.gqa_attn_get_error() == 0
    O_ref, L_ref = oracle.forward_cached(to_f64(q), to_f64(k), to_f64(v), causal=causal, scale=scale)
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
                     f"decode B={B} Hq={Hq} Hkv={Hkv} Sq={Sq} Sk={Sk} D={D} splits={num_splits}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sk", [1, 127, 128, 129, 1000, 4096])
def test_single_token_decode(Sk, D):
    g = gqa()
    _case(g, 2, 8, 2, 1, Sk, D, seed=Sk + D)


@pytest.mark.parametrize("Sq,Hq,Hkv", [(2, 8, 2), (4, 32, 8), (3, 4, 4), (16, 8, 8), (8, 16, 8)])
def test_multi_token_causal(Sq, Hq, Hkv):
    g = gqa()
    _case(g, 1, Hq, Hkv, Sq, 777, 128, seed=Sq * 7 + Hq)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_split_counts_agree(splits):
    """Any number of key chunks gives the same result (the combine is associative)."""
    g = gqa()
    _case(g, 1, 32, 8, 1, 3000, 128, seed=5, num_splits=splits)


def test_non_causal_prefill_over_cache():
    g = gqa()
    _case(g, 2, 12, 4, 4, 600, 64, seed=11, causal=False)


def test_decode_equals_fwd_tail():
    """Decoding the last Sq rows against the cache equals the training forward's last Sq rows."""
    g = gqa()
    B, Hq, Hkv, S, D, Sq = 1, 8, 2, 640, 128, 2
    q, k, v, _ = (t.cuda() if t is not None else None for t in make_inputs(B, Hq, Hkv, S, D, 3, with_do=False))
    o_full, l_full = g.gqa_attn_fwd(q, k, v)
    o, l = g.gqa_attn_decode_fwd(q[:, :, -Sq:].contiguous(), k, v)
    assert (o.float() - o_full[:, :, -Sq:].float()).abs().max().item() <= 1e-2
    assert (l - l_full[:, :, -Sq:]).abs().max().item() <= 1e-3


def test_rejects_too_many_rows():
    g = gqa()
    q = torch.zeros(1, 32, 1, 128, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 64, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(g.GqaAttnError):
        g.gqa_attn_decode_fwd(q, k, k)  # 32 query heads on one KV head: 32 rows > 16


def test_merge_bitwise_reproducible():
    """The CTA that finishes its KV head's last chunk merges every chunk in chunk order, so repeated
    calls give the same bits whichever CTA happens to finish last (many chunks per KV head)."""
    g = gqa()
    _, k, v, _ = make_inputs(2, 16, 4, 4096, 128, 31, with_do=False)
    q = make_inputs(2, 16, 4, 2, 128, 1031, with_do=False)[0]
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    runs = [g.gqa_attn_decode_fwd(q, k, v, num_splits=64) for _ in range(4)]  # 64 chunks of 64 keys
    assert g.gqa_attn_get_error() == 0
    for o, lse in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
