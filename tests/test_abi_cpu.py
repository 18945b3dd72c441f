"""The C ABI without a GPU: the library builds, loads, exports every declared entry point,
and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")
# the stable interface and the hooks of the library's own tests and benchmark
HEADERS = [HEADER, os.path.join(ROOT, "include", "gqa_attn_testing.h")]


def _header_sources():
    return "\n".join(re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S) for h in HEADERS)


def _declared_functions():
    return sorted(set(re.findall(r"\b(gqa_attn_[a-z_]+)\s*\(", _header_sources())))


@pytest.fixture(scope="module")
def lib():
    from causal_gqa_attention_flash_gb300.build import build_library
    from causal_gqa_attention_flash_gb300 import _lib
    build_library()
    return _lib.load()


def test_header_declares_the_boundary():
    stable = re.findall(r"\b(gqa_attn_[a-z_]+)\s*\(", re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S))
    for n in ("gqa_attn_fwd", "gqa_attn_bwd", "gqa_attn_bwd_workspace_size", "gqa_attn_get_error",
              "gqa_attn_strerror"):
        assert n in stable
    # the testing hooks live outside the stable header
    for n in ("gqa_attn_selftest_wait_timeout", "gqa_attn_trace_arm", "gqa_attn_trace_collect"):
        assert n not in stable and n in _declared_functions()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in gqa_attn.h but not exported"


def test_binding_declares_every_symbol():
    from causal_gqa_attention_flash_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == _declared_functions()


def _declared_arities():
    src = _header_sources()
    out = {}
    for name, params in re.findall(r"\b(gqa_attn_[a-z_]+)\s*\(([^)]*)\)\s*;", src):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arities_match_the_header():
    """Each ctypes prototype has as many parameters as the C declaration."""
    from causal_gqa_attention_flash_gb300 import _lib
    arities = _declared_arities()
    assert sorted(arities) == _declared_functions()
    for name, (_, argtypes) in _lib.SIGNATURES.items():
        assert len(argtypes) == arities[name], f"{name}: binding {len(argtypes)} vs header {arities[name]}"


def test_strerror_and_workspace_size(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -99):
        assert isinstance(lib.gqa_attn_strerror(code), bytes)
    assert b"debug build" in lib.gqa_attn_strerror(-7)
    assert lib.gqa_attn_bwd_workspace_size(1, 4, 2, 128, 96) == 0
    assert lib.gqa_attn_bwd_workspace_size(1, 4, 3, 128, 64) == 0
    n = lib.gqa_attn_bwd_workspace_size(2, 32, 8, 16384, 128)
    # D and LSE2 rows (f32, padded to 128) + f32 dQ accumulator + one arrival counter per key tile
    # of each (batch entry, KV head), 256-byte aligned sections; no key tile of this size is split
    assert n == 2 * 2 * 32 * 16384 * 4 + 2 * 32 * 16384 * 128 * 4 + 2 * 8 * 128 * 4
    n = lib.gqa_attn_bwd_workspace_size(1, 4, 2, 130, 64)
    rows_pad = 4 * 256
    assert n >= 2 * rows_pad * 4 + 4 * 130 * 64 * 4 and n % 256 == 0


def test_host_argument_checks_need_no_gpu(lib):
    """Arguments the host rejects return their code before any CUDA call (fake aligned addresses)."""
    A = 1 << 20  # an aligned, never-dereferenced address
    assert lib.gqa_attn_fwd(None, A, A, A, A, 1, 4, 2, 128, 64, 1, 0.125, None) == -1
    assert lib.gqa_attn_fwd(A, A, A, A, A, 1, 4, 3, 128, 64, 1, 0.125, None) == -1
    assert lib.gqa_attn_fwd(A, A, A, A, A, 1, 4, 2, 128, 80, 1, 0.125, None) == -2
    assert lib.gqa_attn_fwd(A + 8, A, A, A, A, 1, 4, 2, 128, 64, 1, 0.125, None) == -1
    assert lib.gqa_attn_fwd(A, A, A, A, A, 1, 4, 2, 128, 64, 1, float("inf"), None) == -1
    assert lib.gqa_attn_fwd(A, A, A, A, A, 0, 4, 2, 128, 64, 1, 0.125, None) == -1
    assert lib.gqa_attn_fwd(A, A, A, A, A, 1, 4, 2, 128 * 65536, 64, 1, 0.125, None) == -2
    args = [A] * 10
    assert lib.gqa_attn_bwd(*args, 0, 1, 4, 2, 128, 64, 1, 0.125, None) == -3
    assert lib.gqa_attn_bwd(*args[:9], A + 128, 1 << 30, 1, 4, 2, 128, 64, 1, 0.125, None) == -1
    assert lib.gqa_attn_selftest_wait_timeout(0, None) == -1


def test_noalloc_returns_the_codes_of_the_workspace_backward(lib):
    """Rejected sizes give the same code from gqa_attn_bwd_noalloc as from gqa_attn_bwd (no CUDA call)."""
    A = 1 << 20
    for (B, Hq, Hkv, S, D, scale, code) in ((1, 4, 2, 128, 96, 0.125, -2), (1, 4, 3, 128, 64, 0.125, -1),
                                             (0, 4, 2, 128, 64, 0.125, -1), (1, 4, 2, 128, 64, float("nan"), -1),
                                             (1, 4, 2, 128 * 65536, 64, 0.125, -2)):
        assert lib.gqa_attn_bwd(*([A] * 10), 1 << 40, B, Hq, Hkv, S, D, 1, scale, None) == code
        assert lib.gqa_attn_bwd_noalloc(*([A] * 9), B, Hq, Hkv, S, D, 1, scale, None) == code
    assert lib.gqa_attn_bwd_noalloc(None, *([A] * 8), 1, 4, 2, 128, 64, 1, 0.125, None) == -1


def test_padded_row_count_is_bounded(lib):
    """B * Hq * (S rounded up to the 128-row tile) indexes the backward's padded rows in 32 bits."""
    A = 1 << 20
    # S = 1 pads to 128 rows: 2^24 heads x 128 rows = 2^31 padded rows, refused
    assert lib.gqa_attn_fwd(A, A, A, A, A, 1 << 12, 1 << 12, 1 << 12, 1, 64, 1, 0.125, None) == -2
    assert lib.gqa_attn_bwd_workspace_size(1 << 12, 1 << 12, 1 << 12, 1, 64) == 0


def _fake_cuda():
    torch = pytest.importorskip("torch")
    from torch._subclasses.fake_tensor import FakeTensorMode
    return torch, FakeTensorMode()


def test_binding_checks_caller_buffers_before_any_launch():
    """Every caller-supplied buffer is checked in Python before the library is called: wrong shape,
    dtype or contiguity of an output raises ValueError (checked on fake CUDA tensors, no GPU)."""
    torch, mode = _fake_cuda()
    import causal_gqa_attention_flash_gb300 as g
    with mode:
        q = torch.empty(1, 4, 128, 64, device="cuda", dtype=torch.bfloat16)
        k = torch.empty(1, 2, 128, 64, device="cuda", dtype=torch.bfloat16)
        lse = torch.empty(1, 4, 128, device="cuda", dtype=torch.float32)
        bad = {
            "dq shape": dict(dq=torch.empty(1, 4, 128, 32, device="cuda", dtype=torch.bfloat16)),
            "dq dtype": dict(dq=torch.empty(1, 4, 128, 64, device="cuda", dtype=torch.float16)),
            "dk shape": dict(dk=torch.empty(1, 4, 128, 64, device="cuda", dtype=torch.bfloat16)),
            "dv strided": dict(dv=torch.empty(1, 2, 64, 128, device="cuda", dtype=torch.bfloat16).transpose(2, 3)),
            "workspace dtype": dict(workspace=torch.empty(1 << 20, device="cuda", dtype=torch.float32)),
        }
        for what, kw in bad.items():
            with pytest.raises(ValueError):
                g.gqa_attn_bwd(q, k, k, q, q, lse, **kw)
        with pytest.raises(ValueError):
            g.gqa_attn_bwd(q, k, k, q, q, torch.empty(1, 4, 127, device="cuda"))  # lse shape
        with pytest.raises(ValueError):
            g.gqa_attn_fwd(q, k, k, o=torch.empty(1, 4, 128, 64, device="cuda", dtype=torch.float32))
        with pytest.raises(ValueError):
            g.gqa_attn_fwd(q, k, k, lse=torch.empty(1, 4, 128, device="cuda", dtype=torch.float64))
        with pytest.raises(ValueError):
            g.gqa_attn_bwd_noalloc(q, k, k, q, q, lse, q, k, torch.empty(1, 2, 128, 32, device="cuda",
                                                                      dtype=torch.bfloat16))
        with pytest.raises(ValueError):
            g.gqa_attn_decode_fwd(q[:, :, :1].contiguous(), k, k, lse=torch.empty(1, 4, 2, device="cuda"))
        with pytest.raises(ValueError):  # CPU output for CUDA inputs
            g.gqa_attn_fwd(q, k, k, o=torch.empty(1, 4, 128, 64, dtype=torch.bfloat16))


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from causal_gqa_attention_flash_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "causal_gqa_attention_flash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle/" not in src, f


def _tile_steps(jt, n_tiles, G, causal):
    return G * (n_tiles - jt if causal else n_tiles)


def _makespan(B, Hkv, G, n_tiles, causal, cap, overhead=4, sms=152):
    import heapq
    sizes = []
    for jt in range(n_tiles):
        st = _tile_steps(jt, n_tiles, G, causal)
        parts = -(-st // cap) if cap else 1
        sizes += [(p + 1) * st // parts - p * st // parts + overhead for p in range(parts)] * (B * Hkv)
    load = [0] * sms
    span = 0
    for sz in sorted(sizes, reverse=True):
        t = heapq.heappop(load) + sz
        heapq.heappush(load, t)
        span = max(span, t)
    return span


def _split_plan(B, Hkv, G, n_tiles, causal):
    """The backward's key-tile split, restated: the cap with the shortest longest-first makespan
    (CTAs cost their steps plus 4), taken if it beats the unsplit grid by 15%; then the parts of
    every key tile with their step ranges. None: nothing is split."""
    steps0 = _tile_steps(0, n_tiles, G, causal)
    if B * Hkv * n_tiles > 2 * 152 or steps0 < 2:
        return None, 0
    unsplit = best = _makespan(B, Hkv, G, n_tiles, causal, 0)
    best_cap = 0
    for cap in range(steps0 - 1, 0, -1):
        if B * Hkv * sum(-(-_tile_steps(jt, n_tiles, G, causal) // cap) for jt in range(n_tiles)) > 4 * 152:
            break  # grids of more than four waves are not considered
        m = _makespan(B, Hkv, G, n_tiles, causal, cap)
        if m < best:
            best, best_cap = m, cap
    if best_cap == 0 or best * 1.15 > unsplit:
        return None, 0
    plan = []
    for jt in range(n_tiles):
        st = _tile_steps(jt, n_tiles, G, causal)
        parts = -(-st // best_cap)
        plan.append((jt, [(p * st // parts, (p + 1) * st // parts) for p in range(parts)]))
    return plan, best_cap


@pytest.mark.parametrize("B,Hq,Hkv,S,causal", [(4, 12, 4, 1024, 1), (8, 8, 2, 512, 1), (1, 32, 8, 4096, 1),
                                               (1, 4, 2, 128, 1), (2, 6, 3, 300, 0), (2, 32, 8, 16384, 1)])
def test_split_parts_cover_every_step_once(B, Hq, Hkv, S, causal):
    """Host logic of the split backward: the parts of a key tile cover its steps exactly once, in
    order, with at most `cap` steps each, and the workspace holds every partial."""
    import math
    G, n_tiles = Hq // Hkv, math.ceil(S / 128)
    plan, cap = _split_plan(B, Hkv, G, n_tiles, causal)
    if plan is None:
        assert (B, Hq, S) not in ((4, 12, 1024), (8, 8, 512)), "the small workloads are expected to split"
        return
    parts_per_group = 0
    for jt, parts in plan:
        steps = G * (n_tiles - jt if causal else n_tiles)
        assert parts[0][0] == 0 and parts[-1][1] == steps
        for (a, b), (c, _) in zip(parts, parts[1:]):
            assert b == c
        assert all(0 < b - a <= cap for a, b in parts)
        if len(parts) > 1:
            parts_per_group += len(parts)
    from causal_gqa_attention_flash_gb300 import _lib
    lib = _lib.load()
    n = lib.gqa_attn_bwd_workspace_size(B, Hq, Hkv, S, 64)
    assert n >= B * Hkv * parts_per_group * 128 * 64 * 2 * 4


def _kv_tiles(qt, Sq, Sk, causal):
    if qt * 128 >= Sq:
        return 0
    if not causal:
        return -(-Sk // 128)
    return (Sk - Sq + min(Sq - 1, qt * 128 + 127)) // 128 + 1


def _fwd_parts(nA, nB, parts):
    n_all = max(nA, nB)
    return [(q * nA // parts, n_all if q == parts - 1 else (q + 1) * nA // parts) for q in range(parts)]


def _fwd_slot_floats(D):
    return 2 * (128 * D + 2 * 128)


def _fwd_split_plan(BH, Sq, Sk, causal, D, sms=152):
    """The forward's key-range split, restated: query-tile pairs (tiles 2p, 2p + 1) whose tile A
    sees more than `cap` key tiles split into ceil(nA / cap) parts. A CTA costs one unit per
    (query tile, key tile) product plus 4, plus 2 for a part of a split pair; CTAs are dealt longest
    first onto 152 SMs; a split adds the merge, 4 units plus one per 3 MiB of slots. The cap with
    the shortest estimate is taken if it beats the unsplit grid by 15%. Returns (cap, slots per
    head, split pairs); cap 0: nothing split."""
    import heapq
    n_pairs = -(-Sq // 256)

    def makespan(cap):
        sizes, slots = [], 0
        for pr in range(n_pairs):
            nA, nB = _kv_tiles(2 * pr, Sq, Sk, causal), _kv_tiles(2 * pr + 1, Sq, Sk, causal)
            if nA == 0:
                continue
            parts = -(-nA // cap) if cap and nA > cap else 1
            if parts > 1:
                slots += parts
            for kb, ke in _fwd_parts(nA, nB, parts):
                sizes += [4 + (2 if parts > 1 else 0) + sum((j < nA) + (j < nB) for j in range(kb, ke))] * BH
        load, span = [0] * sms, 0
        for sz in sorted(sizes, reverse=True):
            t = heapq.heappop(load) + sz
            heapq.heappush(load, t)
            span = max(span, t)
        if slots:
            span += 4 + slots * BH * _fwd_slot_floats(D) * 4 // (3 << 20)
        return span

    nA_max = max(_kv_tiles(0, Sq, Sk, causal), _kv_tiles(2 * (n_pairs - 1), Sq, Sk, causal))
    if BH * n_pairs > 2 * sms or nA_max < 2:
        return 0, 0, 0
    unsplit = best = makespan(0)
    best_cap = 0
    for cap in range(nA_max - 1, 0, -1):
        ctas = sum((-(-nA // cap) if nA > cap else (1 if nA > 0 else 0))
                   for nA in (_kv_tiles(2 * pr, Sq, Sk, causal) for pr in range(n_pairs)))
        if BH * ctas > 4 * sms:
            break  # grids of more than four waves are not considered
        m = makespan(cap)
        if m < best:
            best, best_cap = m, cap
    if best_cap == 0 or best * 1.15 > unsplit:
        return 0, 0, 0
    slots = pairs = 0
    for pr in range(n_pairs):
        nA = _kv_tiles(2 * pr, Sq, Sk, causal)
        if nA > best_cap:
            slots += -(-nA // best_cap)
            pairs += 1
    return best_cap, slots, pairs


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D", [(1, 4, 2, 300, 300, 64), (2, 6, 3, 700, 700, 128),
                                              (1, 8, 2, 512, 4096, 128), (1, 32, 8, 512, 16384, 128),
                                              (2, 32, 8, 2048, 2048, 128), (8, 32, 8, 512, 512, 64)])
def test_forward_split_parts_and_workspace(B, Hq, Hkv, Sq, Sk, D):
    """Host logic of the split forward: each part of a pair holds at least one key tile of tile A
    and at most `cap` of them, the parts cover the pair's key tiles once, in order, and the
    workspace holds one slot per part (two tiles of 128 x D floats, m and l)."""
    from causal_gqa_attention_flash_gb300 import _lib
    lib = _lib.load()
    slots = 0
    for causal in (0, 1):
        cap, s, _ = _fwd_split_plan(B * Hq, Sq, Sk, causal, D)
        slots = max(slots, s)
        for pr in range(-(-Sq // 256)):
            nA, nB = _kv_tiles(2 * pr, Sq, Sk, causal), _kv_tiles(2 * pr + 1, Sq, Sk, causal)
            parts = _fwd_parts(nA, nB, -(-nA // cap) if cap and nA > cap else 1)
            assert parts[0][0] == 0 and parts[-1][1] == max(nA, nB)
            assert all(b == c for (_, b), (c, _) in zip(parts, parts[1:]))
            assert all(min(nA, b) - a >= 1 and (not cap or min(nA, b) - a <= cap) for a, b in parts)
    n = lib.gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, D)
    if slots == 0:
        assert n == 0
        return
    assert n == -(-(B * Hq * slots * _fwd_slot_floats(D) * 4) // 256) * 256
    assert (1, 8, 512, 4096) != (B, Hq, Sq, Sk) or n > 0


def test_split_plans_are_quick_for_long_key_ranges(lib):
    """The split plans search key-range caps on a first call for each size; the search stops at
    four waves, so a very long cache over a small grid plans in well under a second."""
    import time
    t0 = time.perf_counter()
    for B, Hq, Hkv, Sq, Sk in ((1, 1, 1, 128, 1 << 20), (1, 8, 1, 200, 1 << 19), (19, 8, 2, 256, 1 << 18)):
        n = lib.gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, 128)
        assert n % 256 == 0
    lib.gqa_attn_bwd_workspace_size(1, 64, 1, 8192, 64)  # 64 query heads on one KV head: long key tiles
    assert time.perf_counter() - t0 < 2.0
