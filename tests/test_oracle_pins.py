"""The oracle against what the mathematics fixes (CPU only).

Each test runs one pin from ``oracle_checks``; see there for what each pin
compares against.
"""

import numpy as np
import pytest

import oracle
import oracle_checks as oc
from oracle import monoid


def test_decimal_bruteforce():
    oc.check_decimal_bruteforce(oracle)


def test_finite_differences():
    oc.check_finite_differences(oracle)


def test_closed_forms():
    oc.check_closed_forms(oracle)


def test_invariants():
    oc.check_invariants(oracle)


def test_torch_sdpa_f64():
    oc.check_torch_sdpa(oracle)


def test_monoid_regrouping():
    oc.check_monoid_regrouping(oracle, monoid)


def test_row_variants():
    oc.check_row_variants(oracle)


def test_decode_cached_attention():
    oc.check_decode(oracle)


def test_varlen_packed_batches():
    oc.check_varlen(oracle)


def test_rope():
    oc.check_rope(oracle)


def test_golden_file():
    oc.check_golden(oracle)


def test_golden_forward_is_decimal_exact():
    """The stored golden forward agrees with the decimal brute force, not only with the oracle."""
    meta, a = oc.load_golden()
    Ob, Lb = oc.brute_forward_decimal(a["q"], a["k"], a["v"], meta["causal"], meta["scale"])
    assert oc._relerr(a["O"], Ob) <= 1e-14
    assert np.max(np.abs(a["LSE"] - Lb)) <= 1e-13


def test_oracle_has_no_product_imports():
    """The oracle imports nothing from the CUDA package (and vice versa is checked by the ABI test)."""
    import pathlib
    root = pathlib.Path(oracle.__file__).parent
    for f in root.glob("*.py"):
        src = f.read_text()
        assert "causal_gqa_attention_flash_gb300" not in src, f
        assert "ctypes" not in src, f
