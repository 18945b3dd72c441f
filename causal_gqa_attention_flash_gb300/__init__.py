"""Fused causal grouped-query attention (forward + backward) for GB300, sm_103a.

A thin Python binding over the C ABI of ``libgqa_attn.so`` (declared in
``include/gqa_attn.h``). Every function here only marshals arguments:
it checks tensor placement, dtype and shape, allocates outputs with torch
(device memory and streams are the only things torch provides), and calls
the entry point of the same name. All arithmetic runs in the library's CUDA
kernels; if the library is missing, the call raises.

    o, lse = gqa_attn_fwd(q, k, v, causal=True)
    dq, dk, dv = gqa_attn_bwd(q, k, v, o, dO, lse, causal=True)

Layout is BHSD: q, o, dO, dq are [B, Hq, S, D] bf16; k, v, dk, dv are
[B, Hkv, S, D] bf16; lse is [B, Hq, S] float32. Query head h reads KV head
h // (Hq // Hkv).

Every tensor the caller passes, inputs and outputs alike, is checked before
the call: contiguous, of the expected dtype and shape, on the device of q;
the call then runs with that device current.
"""

from __future__ import annotations

import math

import torch

from . import _lib

__all__ = [
    "GqaAttnError",
    "gqa_attn_fwd",
    "gqa_attn_bwd",
    "gqa_attn_bwd_workspace_size",
    "gqa_attn_get_error",
    "gqa_attn_strerror",
    "gqa_attn_last_cuda_error",
    "gqa_attn_selftest_wait_timeout",
    "gqa_attn_trace_arm",
    "gqa_attn_trace_collect",
    "gqa_attn_bwd_noalloc",
    "gqa_attn_decode_fwd",
    "gqa_attn_fwd_cached",
    "gqa_attn_fwd_splitkv",
    "gqa_attn_fwd_splitkv_workspace_size",
    "gqa_attn_fwd_varlen",
    "gqa_attn_bwd_varlen",
    "gqa_attn_bwd_varlen_workspace_size",
    "gqa_attn_fwd_rope",
    "gqa_attn_bwd_rope",
    "gqa_attn_fwd_rope_workspace_size",
    "gqa_attn_bwd_rope_workspace_size",
    "gqa_attn_decode_workspace_size",
    "NOALLOC_SCRATCH_BYTES",
    "KERNEL_NAMES",
    "lib_path",
]

# Tracing slots in the header's GQA_KERNEL_* order. "decode_combine" is no longer launched (the last
# split CTA of each KV head merges the chunks); its slot stays so that the numbering is stable.
KERNEL_NAMES = ("fwd", "bwd_prep", "bwd_main", "bwd_convert", "decode_split", "decode_combine", "bwd_dkdv", "bwd_dq", "rope",
                "fwd_combine")

GQA_OK = 0
GQA_ERR_INVALID_ARG = -1
GQA_ERR_UNSUPPORTED = -2
GQA_ERR_WORKSPACE_TOO_SMALL = -3
GQA_ERR_CUDA = -4
GQA_ERR_TIMEOUT = -5
GQA_ERR_INTERNAL = -6
GQA_ERR_BOUNDS = -7
NOALLOC_SCRATCH_BYTES = 64 << 20  # GQA_NOALLOC_SCRATCH_BYTES of include/gqa_attn.h


class GqaAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = gqa_attn_strerror(code)
        if code == GQA_ERR_CUDA:
            msg += f" (cudaError {gqa_attn_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")
        self.code = code


def lib_path() -> str:
    return _lib.LIB_PATH


def gqa_attn_strerror(code: int) -> str:
    return _lib.load().gqa_attn_strerror(int(code)).decode()


def gqa_attn_last_cuda_error() -> int:
    return int(_lib.load().gqa_attn_last_cuda_error())


def _stream_handle(stream, device=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def _check(rc: int, where: str) -> None:
    if rc != GQA_OK:
        raise GqaAttnError(rc, where)


def _want(name, t, shape, dtype, device):
    """A caller-supplied tensor must be contiguous, of the given dtype and shape, on `device`:
    the library writes through its pointer, so a mismatch is refused here, before any launch."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if (not t.is_cuda or t.device != device or t.dtype != dtype or tuple(t.shape) != tuple(shape)
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor of shape {tuple(shape)} on {device}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}"
                         + ("" if t.is_contiguous() else " (not contiguous)"))
    return t


def _out(name, t, shape, dtype, device):
    """Output buffer: the caller's (checked) or a new one."""
    if t is None:
        return torch.empty(tuple(shape), device=device, dtype=dtype)
    return _want(name, t, shape, dtype, device)


def _workspace(t, need, device):
    """Workspace buffer: the caller's (a contiguous uint8 CUDA tensor on `device`; its size is
    checked by the library) or a new one of `need` bytes."""
    if t is None:
        return torch.empty(max(int(need), 256), device=device, dtype=torch.uint8)
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device or t.dtype != torch.uint8
            or not t.is_contiguous()):
        raise ValueError(f"workspace must be a contiguous uint8 CUDA tensor on {device}")
    return t


def _dims(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bfloat16 CUDA tensor (BHSD), got "
                             f"{getattr(t, 'dtype', None)} {tuple(getattr(t, 'shape', ()))} on "
                             f"{getattr(t, 'device', None)}")
    B, Hq, S, D = q.shape
    if k.shape[0] != B or k.shape[2] != S or k.shape[3] != D or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if k.device != q.device or v.device != q.device:
        raise ValueError(f"q, k, v must be on one device, got {q.device}, {k.device}, {v.device}")
    return B, Hq, k.shape[1], S, D


def gqa_attn_fwd(q, k, v, causal: bool = True, scale: float | None = None, o=None, lse=None, stream=None):
    """Forward: returns (o [B,Hq,S,D] bf16, lse [B,Hq,S] f32). ``scale`` defaults to 1/sqrt(D)."""
    B, Hq, Hkv, S, D = _dims(q, k, v)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (B, Hq, S), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      B, Hq, Hkv, S, D, int(bool(causal)), float(scale), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_fwd")
    return o, lse


def gqa_attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, S: int, D: int) -> int:
    return int(_lib.load().gqa_attn_bwd_workspace_size(B, Hq, Hkv, S, D))


def gqa_attn_bwd(q, k, v, o, dO, lse, causal: bool = True, scale: float | None = None,
                 dq=None, dk=None, dv=None, workspace=None, stream=None, deterministic: bool = False):
    """Backward of sum(o * dO): returns (dq, dk, dv), bf16, shaped like q, k, v.

    ``workspace`` (optional) is a uint8 CUDA tensor of at least
    ``gqa_attn_bwd_workspace_size(...)`` bytes; one is allocated if omitted.
    ``deterministic`` selects gqa_attn_bwd_deterministic (bitwise reproducible dQ).
    """
    B, Hq, Hkv, S, D = _grad_inputs(q, k, v, o, dO, lse)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = _out("dq", dq, q.shape, torch.bfloat16, dev)
    dk = _out("dk", dk, k.shape, torch.bfloat16, dev)
    dv = _out("dv", dv, v.shape, torch.bfloat16, dev)
    workspace = _workspace(workspace, gqa_attn_bwd_workspace_size(B, Hq, Hkv, S, D), dev)
    nbytes = workspace.numel() * workspace.element_size()
    name = "gqa_attn_bwd_deterministic" if deterministic else "gqa_attn_bwd"
    with torch.cuda.device(dev):
        rc = getattr(_lib.load(), name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
                                        lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                        workspace.data_ptr(), nbytes, B, Hq, Hkv, S, D, int(bool(causal)),
                                        float(scale), _stream_handle(stream, dev))
    _check(rc, name)
    return dq, dk, dv


def _grad_inputs(q, k, v, o, dO, lse):
    """Checks of a backward's inputs: q, k, v as the forward's, o and dO shaped like q, lse [B, Hq, S]."""
    B, Hq, Hkv, S, D = _dims(q, k, v)
    _want("o", o, q.shape, torch.bfloat16, q.device)
    _want("dO", dO, q.shape, torch.bfloat16, q.device)
    _want("lse", lse, (B, Hq, S), torch.float32, q.device)
    return B, Hq, Hkv, S, D


def gqa_attn_get_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) its status word on the current device: 0 or a
    negative code raised by kernels launched on that stream."""
    return int(_lib.load().gqa_attn_get_error(_stream_handle(stream)))


def gqa_attn_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nothing ends; it gives up after limit_us).
    A testing hook (gqa_attn_testing.h), not part of the stable interface."""
    _check(_lib.load().gqa_attn_selftest_wait_timeout(int(limit_us), _stream_handle(stream)),
           "gqa_attn_selftest_wait_timeout")


def gqa_attn_trace_arm() -> None:
    """Arm per-kernel event timing for the following calls on this host thread."""
    _check(_lib.load().gqa_attn_trace_arm(), "gqa_attn_trace_arm")


def gqa_attn_trace_collect() -> dict:
    """Disarm and return {kernel name: (launches, total ms)} of the calls since arming."""
    import ctypes
    n = len(KERNEL_NAMES)
    launches = (ctypes.c_int * n)()
    total = (ctypes.c_double * n)()
    _check(_lib.load().gqa_attn_trace_collect(launches, total), "gqa_attn_trace_collect")
    return {name: (int(launches[i]), float(total[i])) for i, name in enumerate(KERNEL_NAMES)}


def gqa_attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, causal: bool = True, scale: float | None = None,
                         stream=None):
    """Backward into caller-provided dq, dk, dv using the library's static scratch array.

    For callers that cannot allocate device memory: nothing is allocated here
    or in the library (the outputs must be given). The scratch array holds
    NOALLOC_SCRATCH_BYTES; larger problems raise GqaAttnError (workspace too
    small). Calls that overlap on the GPU race on the shared array.
    """
    B, Hq, Hkv, S, D = _grad_inputs(q, k, v, o, dO, lse)
    dev = q.device
    _want("dq", dq, q.shape, torch.bfloat16, dev)
    _want("dk", dk, k.shape, torch.bfloat16, dev)
    _want("dv", dv, v.shape, torch.bfloat16, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                              dO.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                              dv.data_ptr(), B, Hq, Hkv, S, D, int(bool(causal)), float(scale),
                                              _stream_handle(stream, dev))
    _check(rc, "gqa_attn_bwd_noalloc")
    return dq, dk, dv


def gqa_attn_decode_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, num_splits: int = 0) -> int:
    return int(_lib.load().gqa_attn_decode_workspace_size(B, Hq, Hkv, Sq, Sk, D, num_splits))


def gqa_attn_decode_fwd(q, k_cache, v_cache, causal: bool = True, scale: float | None = None, num_splits: int = 0,
                        o=None, lse=None, workspace=None, stream=None):
    """Attention of q [B,Hq,Sq,D] against a cache k/v [B,Hkv,Sk,D] (Sq <= Sk, query i at position
    Sk - Sq + i). Returns (o [B,Hq,Sq,D] bf16, lse [B,Hq,Sq] f32)."""
    B, Hq, Hkv, Sq, Sk, D = _cache_dims(q, k_cache, v_cache)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (B, Hq, Sq), torch.float32, dev)
    workspace = _workspace(workspace, gqa_attn_decode_workspace_size(B, Hq, Hkv, Sq, Sk, D, num_splits), dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_decode_fwd(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr(),
                                             lse.data_ptr(), workspace.data_ptr(), nbytes, B, Hq, Hkv, Sq, Sk, D,
                                             int(bool(causal)), float(scale), int(num_splits),
                                             _stream_handle(stream, dev))
    _check(rc, "gqa_attn_decode_fwd")
    return o, lse


def gqa_attn_fwd_cached(q, k_cache, v_cache, causal: bool = True, scale: float | None = None, o=None, lse=None,
                        stream=None):
    """Forward of q [B,Hq,Sq,D] over k/v [B,Hkv,Sk,D] (Sq <= Sk, query r at position Sk - Sq + r),
    on the tensor cores. Returns (o [B,Hq,Sq,D] bf16, lse [B,Hq,Sq] f32)."""
    B, Hq, Hkv, Sq, Sk, D = _cache_dims(q, k_cache, v_cache)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (B, Hq, Sq), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_fwd_cached(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr(),
                                             lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), float(scale),
                                             _stream_handle(stream, dev))
    _check(rc, "gqa_attn_fwd_cached")
    return o, lse


def gqa_attn_fwd_splitkv_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int) -> int:
    """Bytes of workspace gqa_attn_fwd_splitkv needs (0: these sizes are never split)."""
    return int(_lib.load().gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, D))


def gqa_attn_fwd_splitkv(q, k_cache, v_cache, causal: bool = True, scale: float | None = None, o=None, lse=None,
                         workspace=None, stream=None):
    """Forward of q [B,Hq,Sq,D] over k/v [B,Hkv,Sk,D] (Sq <= Sk; Sq = Sk is the training forward)
    whose key range is split across CTAs when the grid is small. Returns (o, lse) like
    gqa_attn_fwd_cached; ``workspace`` (optional) is a uint8 CUDA tensor of at least
    ``gqa_attn_fwd_splitkv_workspace_size(...)`` bytes."""
    B, Hq, Hkv, Sq, Sk, D = _cache_dims(q, k_cache, v_cache)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (B, Hq, Sq), torch.float32, dev)
    need = gqa_attn_fwd_splitkv_workspace_size(B, Hq, Hkv, Sq, Sk, D)
    ws_ptr, nbytes = 0, 0
    if need > 0 or workspace is not None:
        workspace = _workspace(workspace, need, dev)
        ws_ptr, nbytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_fwd_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr(),
                                              lse.data_ptr(), ws_ptr or None, nbytes, B, Hq, Hkv, Sq, Sk, D,
                                              int(bool(causal)), float(scale), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_fwd_splitkv")
    return o, lse


def _cache_dims(q, k_cache, v_cache):
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous 4-D bfloat16 CUDA tensor (BHSD)")
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Hkv, Sk, D) or v_cache.shape != k_cache.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k_cache.shape)}, v {tuple(v_cache.shape)}")
    if k_cache.device != q.device or v_cache.device != q.device:
        raise ValueError("q, k_cache, v_cache must be on one device")
    return B, Hq, Hkv, Sq, Sk, D


def _check_packed(name, t):
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous 3-D bfloat16 CUDA tensor ([H, T, D])")


def _check_cu(name, cu, device):
    if not isinstance(cu, torch.Tensor) or not cu.is_cuda or cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_contiguous() or cu.numel() < 2:
        raise ValueError(f"{name} must be a contiguous 1-D int32 CUDA tensor of nseq + 1 bounds")
    if cu.device != device:
        raise ValueError(f"{name} is on {cu.device}, the tensors on {device}")


def gqa_attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool = True,
                        scale: float | None = None, o=None, lse=None, stream=None):
    """Forward of a packed batch: q [Hq, Tq, D], k/v [Hkv, Tk, D], sequence i owning query rows
    cu_seqlens_q[i]:cu_seqlens_q[i+1] and key rows cu_seqlens_k[i]:cu_seqlens_k[i+1] (int32 CUDA
    tensors). Returns (o [Hq, Tq, D] bf16, lse [Hq, Tq] f32)."""
    _check_packed("q", q)
    _check_packed("k", k)
    _check_packed("v", v)
    Hq, Tq, D = q.shape
    Hkv, Tk = k.shape[0], k.shape[1]
    if k.shape != (Hkv, Tk, D) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    dev = q.device
    if k.device != dev or v.device != dev:
        raise ValueError("q, k, v must be on one device")
    _check_cu("cu_seqlens_q", cu_seqlens_q, dev)
    _check_cu("cu_seqlens_k", cu_seqlens_k, dev)
    if cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must describe the same number of sequences")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (Hq, Tq), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                             cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                             cu_seqlens_q.numel() - 1, int(max_seqlen_q), Hq, Hkv, Tq, Tk, D,
                                             int(bool(causal)), float(scale), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_fwd_varlen")
    return o, lse


def gqa_attn_bwd_varlen_workspace_size(Hq: int, Hkv: int, T: int, D: int) -> int:
    """Bytes of device workspace gqa_attn_bwd_varlen needs (0 for unsupported sizes)."""
    return int(_lib.load().gqa_attn_bwd_varlen_workspace_size(Hq, Hkv, T, D))


def gqa_attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, max_seqlen: int, causal: bool = True,
                        scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of packed self-attention (q, o, dO [Hq, T, D], k, v [Hkv, T, D], lse [Hq, T], int32
    CUDA bounds cu_seqlens): returns (dq, dk, dv), bf16, shaped like q, k, v."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO)):
        _check_packed(name, t)
    Hq, T, D = q.shape
    Hkv = k.shape[0]
    if k.shape != (Hkv, T, D) or v.shape != k.shape or o.shape != q.shape or dO.shape != q.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}, "
                         f"o {tuple(o.shape)}, dO {tuple(dO.shape)}")
    dev = q.device
    for name, t in (("k", k), ("v", v), ("o", o), ("dO", dO)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")
    _want("lse", lse, (Hq, T), torch.float32, dev)
    _check_cu("cu_seqlens", cu_seqlens, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = _out("dq", dq, q.shape, torch.bfloat16, dev)
    dk = _out("dk", dk, k.shape, torch.bfloat16, dev)
    dv = _out("dv", dv, v.shape, torch.bfloat16, dev)
    workspace = _workspace(workspace, gqa_attn_bwd_varlen_workspace_size(Hq, Hkv, T, D), dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
                                             lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                             cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, int(max_seqlen),
                                             workspace.data_ptr(), nbytes, Hq, Hkv, T, D, int(bool(causal)),
                                             float(scale), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_bwd_varlen")
    return dq, dk, dv


def _check_tables(cos, sin, S, D, device):
    for name, t in (("rope_cos", cos), ("rope_sin", sin)):
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32
                or tuple(t.shape) != (S, D // 2) or not t.is_contiguous() or t.device != device):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor [S, D/2] = [{S}, {D // 2}]")


def gqa_attn_fwd_rope_workspace_size(B: int, Hkv: int, S: int, D: int) -> int:
    """Bytes of device workspace gqa_attn_fwd_rope needs (the rotated keys; 0 for unsupported sizes)."""
    return int(_lib.load().gqa_attn_fwd_rope_workspace_size(B, Hkv, S, D))


def gqa_attn_bwd_rope_workspace_size(B: int, Hq: int, Hkv: int, S: int, D: int) -> int:
    """Bytes of device workspace gqa_attn_bwd_rope needs (0 for unsupported sizes)."""
    return int(_lib.load().gqa_attn_bwd_rope_workspace_size(B, Hq, Hkv, S, D))


def gqa_attn_fwd_rope(q, k, v, rope_cos, rope_sin, causal: bool = True, scale: float | None = None, o=None,
                      lse=None, workspace=None, stream=None):
    """Forward over rotary-embedded q and k (rotate-half pairing, f32 tables [S, D/2]):
    returns (o, lse) like gqa_attn_fwd."""
    B, Hq, Hkv, S, D = _dims(q, k, v)
    dev = q.device
    _check_tables(rope_cos, rope_sin, S, D, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = _out("o", o, q.shape, torch.bfloat16, dev)
    lse = _out("lse", lse, (B, Hq, S), torch.float32, dev)
    workspace = _workspace(workspace, gqa_attn_fwd_rope_workspace_size(B, Hkv, S, D), dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), rope_cos.data_ptr(),
                                           rope_sin.data_ptr(), o.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                                           nbytes, B, Hq, Hkv, S, D, int(bool(causal)), float(scale),
                                           _stream_handle(stream, dev))
    _check(rc, "gqa_attn_fwd_rope")
    return o, lse


def gqa_attn_bwd_rope(q, k, v, o, dO, lse, rope_cos, rope_sin, causal: bool = True, scale: float | None = None,
                      dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of the rotary-embedded forward: (dq, dk, dv) with respect to the unrotated q, k."""
    B, Hq, Hkv, S, D = _grad_inputs(q, k, v, o, dO, lse)
    dev = q.device
    _check_tables(rope_cos, rope_sin, S, D, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = _out("dq", dq, q.shape, torch.bfloat16, dev)
    dk = _out("dk", dk, k.shape, torch.bfloat16, dev)
    dv = _out("dv", dv, v.shape, torch.bfloat16, dev)
    workspace = _workspace(workspace, gqa_attn_bwd_rope_workspace_size(B, Hq, Hkv, S, D), dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        rc = _lib.load().gqa_attn_bwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
                                           lse.data_ptr(), rope_cos.data_ptr(), rope_sin.data_ptr(), dq.data_ptr(),
                                           dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), nbytes, B, Hq, Hkv, S,
                                           D, int(bool(causal)), float(scale), _stream_handle(stream, dev))
    _check(rc, "gqa_attn_bwd_rope")
    return dq, dk, dv
