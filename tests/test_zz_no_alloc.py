"""The allocation-free backward entry point, checked against the ordinary one.

Some callers cannot call cudaMalloc (allocation forbidden inside their own
allocator callbacks, frameworks that own all device memory, hosts that must
not allocate after start-up). gqa_attn_bwd_noalloc serves them with a static
device scratch array. This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes on its
own in a fresh process (the first call sets the array up).
"""

import pytest
import torch

from gpu_helpers import TOL_GRAD_ABS_FLOOR, TOL_GRAD_REL, gqa
from gqa_inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _close(a, b):
    a, b = a.float(), b.float()
    return (a - b).abs().max().item() <= TOL_GRAD_REL * b.abs().max().item() + TOL_GRAD_ABS_FLOOR


@pytest.mark.parametrize("name", ["lm101m", "tiny"])
def test_noalloc_matches_workspace_backward_twice(name):
    g = gqa()
    w = WORKLOADS[name]
    q, k, v, dO = (t.cuda() for t in make_inputs(w.B, w.Hq, w.Hkv, w.S, w.D, w.seed, w.do_std))
    o, lse = g.gqa_attn_fwd(q, k, v, causal=True, scale=w.scale)
    ref = g.gqa_attn_bwd(q, k, v, o, dO, lse, causal=True, scale=w.scale)
    for _ in range(2):  # two calls in a row share (and must fully rewrite) the scratch array
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        g.gqa_attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, causal=True, scale=w.scale)
        assert g.gqa_attn_get_error() == 0
        for got, want in zip((dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all()
            assert _close(got, want)
        # dK/dV take the same deterministic path: bitwise equal to the workspace call
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    g = gqa()
    w = WORKLOADS["qwen3_8b"]
    need = g.gqa_attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.S, w.D)
    assert need > g.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(w.B, w.Hq, w.S, w.D, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(w.B, w.Hkv, w.S, w.D, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(w.B, w.Hq, w.S, device="cuda", dtype=torch.float32)
    with pytest.raises(g.GqaAttnError) as ei:
        g.gqa_attn_bwd_noalloc(q, k, k, q, q, lse, q, k, k)
    assert ei.value.code == g.GQA_ERR_WORKSPACE_TOO_SMALL
