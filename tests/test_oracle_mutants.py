"""Planted mistakes in a copy of the oracle, on the CPU: each must fail at least one pin.

Every mutant is the oracle's own source with one plausible mistake
substituted (a wrong head mapping, an off-by-one mask, a dropped scale, a
wrong sign, a transposed operand, ...). A pin set that let one of them
through would not be pinning that part of the oracle.
"""

import pathlib
import types

import pytest

import oracle
import oracle_checks as oc
from oracle import monoid

SRC = (pathlib.Path(oracle.__file__).parent / "attention.py").read_text()
DECODE_SRC = (pathlib.Path(oracle.__file__).parent / "decode.py").read_text()
VARLEN_SRC = (pathlib.Path(oracle.__file__).parent / "varlen.py").read_text()
ROPE_SRC = (pathlib.Path(oracle.__file__).parent / "rope.py").read_text()

MUTANTS = {
    "gqa_head_mapping_modulo": ("return h // (Hq // Hkv)", "return h % Hkv"),
    "causal_sees_next_key": ("np.where(j <= np.asarray(row_idx)[:, None]", "np.where(j <= np.asarray(row_idx)[:, None] + 1"),
    "score_scale_dropped": ("s = scale * (q_rows @ k_head.T)", "s = (q_rows @ k_head.T)"),
    "lse_base2": ("lse = m + np.log(", "lse = m + np.log2("),
    "dS_sign": ("dS = P * (dP - Dvec[:, None])", "dS = P * (dP + Dvec[:, None])"),
    "D_from_dO_only": ("Dvec = (dO[b, h] * O).sum(axis=1)", "Dvec = (dO[b, h] * dO[b, h]).sum(axis=1)"),
    "dQ_transposed_dS": ("dQ[b, h] = scale * (dS @ k[b, g])", "dQ[b, h] = scale * (dS.T @ k[b, g])"),
    "dK_scale_dropped": ("dK[b, g] += scale * (dS.T @ q[b, h])", "dK[b, g] += (dS.T @ q[b, h])"),
    "dK_wrong_q_head": ("dK[b, g] += scale * (dS.T @ q[b, h])", "dK[b, g] += scale * (dS.T @ q[b, g])"),
    "dV_not_summed_over_group": ("dV[b, g] += P.T @ dO[b, h]", "dV[b, g] = P.T @ dO[b, h]"),
    "dV_untransposed_P": ("dV[b, g] += P.T @ dO[b, h]", "dV[b, g] += P @ dO[b, h]"),
    "dkdv_rows_skips_rows": ("first = int(J.min()) if causal else 0", "first = int(J.max()) if causal else 0"),
    "dq_rows_drops_D": ("dP = dO[b, h, rows] @ v[b, g].T\n    Dvec = (dO[b, h, rows] * O).sum(axis=1)",
                        "dP = dO[b, h, rows] @ v[b, g].T\n    Dvec = 0.0 * (dO[b, h, rows] * O).sum(axis=1)"),
}


DECODE_MUTANTS = {
    "decode_top_left_alignment": ("rows = (Sk - Sq) + np.arange(Sq)", "rows = np.arange(Sq)"),
    "decode_off_by_one_position": ("rows = (Sk - Sq) + np.arange(Sq)", "rows = (Sk - Sq - 1) + np.arange(Sq)"),
}


VARLEN_MUTANTS = {
    "varlen_keys_of_earlier_sequences": ("k[None, :, k0:k1], v[None, :, k0:k1]", "k[None, :, :k1], v[None, :, :k1]"),
    "varlen_key_bounds_from_queries": ("q0, q1, k0, k1 = cq[i], cq[i + 1], ck[i], ck[i + 1]",
                                       "q0, q1, k0, k1 = cq[i], cq[i + 1], cq[i], cq[i + 1]"),
    "varlen_backward_always_causal": ("dO[None, :, s0:s1],\n                              causal=causal",
                                      "dO[None, :, s0:s1],\n                              causal=True"),
    "varlen_backward_drops_last_sequence": ("    for i in range(len(cu) - 1):", "    for i in range(len(cu) - 2):"),
}


ROPE_MUTANTS = {
    "rope_interleaved_pairs": ("lo, hi = x[..., :h], x[..., h:]", "lo, hi = x[..., 0::2], x[..., 1::2]"),
    "rope_sin_sign": ("lo * c - hi * s, hi * c + lo * s", "lo * c + hi * s, hi * c - lo * s"),
    "rope_gradient_not_turned_back": ("return unrotate(gq, cos, sin), unrotate(gk, cos, sin), gv",
                                      "return gq, gk, gv"),
    "rope_turned_back_the_wrong_way": ("return rotate(g, cos, -np.asarray(sin, dtype=np.float64))",
                                       "return rotate(g, cos, np.asarray(sin, dtype=np.float64))"),
    "rope_values_rotated": ("return forward(rotate(q, cos, sin), rotate(k, cos, sin), v,",
                            "return forward(rotate(q, cos, sin), rotate(k, cos, sin), rotate(v, cos, sin),"),
}


def _mutant_module(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, f"mutation anchor for {name} not found in the oracle source"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(SRC.replace(old, new, 1), f"<mutant {name}>", "exec"), mod.__dict__)
    mod.forward_cached = oracle.forward_cached
    mod.forward_varlen = oracle.forward_varlen
    mod.backward_varlen = oracle.backward_varlen
    mod.rope, mod.forward_rope, mod.backward_rope = oracle.rope, oracle.forward_rope, oracle.backward_rope
    return mod


def _decode_mutant_module(name):
    """The real attention oracle with a mutated copy of the cached (decode) oracle."""
    old, new = DECODE_MUTANTS[name]
    assert DECODE_SRC.count(old) == 1
    src = DECODE_SRC.replace(old, new, 1).replace("from .attention import", "from oracle.attention import")
    dmod = types.ModuleType(f"oracle_decode_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), dmod.__dict__)
    mod = types.ModuleType(f"oracle_with_{name}")
    mod.__dict__.update({k: getattr(oracle, k) for k in ("forward", "backward", "forward_rows",
                                                          "backward_dq_rows", "backward_dkdv_rows")})
    mod.forward_cached = dmod.forward_cached
    mod.forward_varlen = oracle.forward_varlen
    mod.backward_varlen = oracle.backward_varlen
    mod.rope, mod.forward_rope, mod.backward_rope = oracle.rope, oracle.forward_rope, oracle.backward_rope
    return mod


def _varlen_mutant_module(name):
    """The real oracle with a mutated copy of the packed variable-length oracle."""
    old, new = VARLEN_MUTANTS[name]
    assert VARLEN_SRC.count(old) == 1, f"mutation anchor for {name} not found"
    src = (VARLEN_SRC.replace(old, new, 1).replace("from .attention import", "from oracle.attention import")
           .replace("from .decode import", "from oracle.decode import"))
    vmod = types.ModuleType(f"oracle_varlen_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), vmod.__dict__)
    mod = types.ModuleType(f"oracle_with_{name}")
    mod.__dict__.update({k: getattr(oracle, k) for k in ("forward", "backward", "forward_rows", "forward_cached",
                                                          "backward_dq_rows", "backward_dkdv_rows")})
    mod.forward_varlen = vmod.forward_varlen
    mod.backward_varlen = vmod.backward_varlen
    return mod


def _first_failing_check(mod):
    for check in oc.ALL_CHECKS:
        fn = getattr(oc, check)
        try:
            if check == "check_monoid_regrouping":
                fn(mod, monoid)
            else:
                fn(mod)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            return check
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    mod = _mutant_module(name)
    caught_by = _first_failing_check(mod)
    assert caught_by is not None, f"no pin catches the planted mistake {name!r}"


@pytest.mark.parametrize("name", sorted(DECODE_MUTANTS))
def test_planted_decode_mistake_is_caught(name):
    mod = _decode_mutant_module(name)
    with pytest.raises(AssertionError):
        oc.check_decode(mod)


@pytest.mark.parametrize("name", sorted(VARLEN_MUTANTS))
def test_planted_varlen_mistake_is_caught(name):
    mod = _varlen_mutant_module(name)
    with pytest.raises(AssertionError):
        oc.check_varlen(mod)


def _rope_mutant_module(name):
    """The real oracle with a mutated copy of the rotary-embedding oracle."""
    old, new = ROPE_MUTANTS[name]
    assert ROPE_SRC.count(old) == 1, f"mutation anchor for {name} not found"
    src = ROPE_SRC.replace(old, new, 1).replace("from .attention import", "from oracle.attention import")
    rmod = types.ModuleType(f"oracle_rope_mutant_{name}")
    exec(compile(src, f"<mutant {name}>", "exec"), rmod.__dict__)
    mod = types.ModuleType(f"oracle_with_{name}")
    mod.rope = rmod
    mod.forward_rope = rmod.forward_rope
    mod.backward_rope = rmod.backward_rope
    return mod


@pytest.mark.parametrize("name", sorted(ROPE_MUTANTS))
def test_planted_rope_mistake_is_caught(name):
    mod = _rope_mutant_module(name)
    with pytest.raises(AssertionError):
        oc.check_rope(mod)
