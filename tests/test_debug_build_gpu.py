"""The checking build (GQA_DEBUG): every kernel checks each computed TMA coordinate and global
index against the extent of the tensor it addresses and reports a failed check as
GQA_ERR_BOUNDS instead of touching memory out of range. It stands in for a memory checker of the
kernels' index arithmetic (compute-sanitizer is not available here).

The parity cases most likely to expose index mistakes -- ragged lengths around the 128-row tile,
packed batches of mixed lengths (sequences starting at any row), split-KV decode, the
deterministic backward and the rotary variants -- run in a child process that loads the checking
build; every one of them asserts a zero status after its calls, so a single failed check fails
the run.
"""

import os
import subprocess
import sys

import pytest

from gpu_helpers import gqa

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    "tests/test_parity_gpu.py::test_ragged_lengths",
    "tests/test_parity_gpu.py::test_non_causal",
    "tests/test_varlen_gpu.py::test_packed_self_attention",
    "tests/test_varlen_gpu.py::test_packed_queries_over_caches",
    "tests/test_varlen_gpu.py::test_packed_backward",
    "tests/test_decode_gpu.py::test_single_token_decode",
    "tests/test_decode_gpu.py::test_multi_token_causal",
    "tests/test_decode_gpu.py::test_split_counts_agree",
    "tests/test_fwd_cached_gpu.py::test_causal_prefill_over_cache",
    "tests/test_fwd_cached_gpu.py::test_splitkv_forward",
    "tests/test_deterministic_gpu.py::test_deterministic_parity",
    "tests/test_rope_gpu.py::test_rope_parity",
]


def test_parity_cases_under_the_checking_build():
    gqa()  # skips without a GPU
    from causal_gqa_attention_flash_gb300.build import build_library
    build_library(debug=True)
    env = dict(os.environ, GQA_ATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *CASES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout

