"""Seeded synthetic inputs for causal grouped-query attention.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It draws random tensors and nothing else: it holds none of the
attention arithmetic.

Workload shapes follow the attention shapes named on the pages:

* ``tiny``      -- B=1, Hq=4,  Hkv=2, S=128,   D=64  (small case, seed 0)
* ``lm101m``    -- B=4, Hq=12, Hkv=4, S=1024,  D=64  ("GQA 12/4 heads, head_dim 64"
  of the 101.7M-parameter dense transformer, RustingBrain docs, "Where it
  stands against PyTorch and TensorFlow"; seed 1)
* ``block512``  -- B=8, Hq=8,  Hkv=2, S=512,   D=64  (``.heads(8, 2, 64)`` of the
  RustingBrain docs, "A language model in twenty lines", at the seq-512
  transformer block of the tang page, "A transformer"; seed 2)
* ``qwen3_8b``  -- B=1, Hq=32, Hkv=8, S=4096,  D=128 (Qwen3-8B-style prefill
  attention, tang page "An LLM"; seed 3)
* ``long16k``   -- B=2, Hq=32, Hkv=8, S=16384, D=128 (long-context training;
  seed 4)

Recipe (one generator per workload): ``torch.Generator('cpu').manual_seed(seed)``;
draw Q, K, V, dO in that order as float32 ``randn`` of their full shapes;
multiply dO by ``do_std`` (0.1, i.e. N(0, 1e-2) read as a variance; 1.0 for
the tiny case); round each to bfloat16 (round-to-nearest-even). The same
bfloat16 bits feed the GPU path and the oracle.

Rotary-position tables (``rope_tables``) are inputs too: cos and sin of
position times base^(-2i/D), the table a caller hands to the RoPE entry points.

Packed batches of variable-length sequences (``make_packed_inputs``) lay the
sequences end to end along the token axis, one [H, T, D] tensor per operand;
the lengths are given, or drawn by ``draw_lengths`` (uniform on [lo, hi] with
its own generator), and the bounds are their running sums starting at 0.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    seed: int
    do_std: float
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def shape_dict(self) -> dict:
        return dict(B=self.B, Hq=self.Hq, Hkv=self.Hkv, S=self.S, D=self.D)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 2, 128, 64, seed=0, do_std=1.0),
    "lm101m": Workload("lm101m", 4, 12, 4, 1024, 64, seed=1, do_std=0.1),
    "block512": Workload("block512", 8, 8, 2, 512, 64, seed=2, do_std=0.1),
    "qwen3_8b": Workload("qwen3_8b", 1, 32, 8, 4096, 128, seed=3, do_std=0.1),
    "long16k": Workload("long16k", 2, 32, 8, 16384, 128, seed=4, do_std=0.1),
}


def make_inputs(B: int, Hq: int, Hkv: int, S: int, D: int, seed: int,
                do_std: float = 0.1, with_do: bool = True):
    """Return bf16 CPU tensors (q, k, v, dO) in BHSD layout, drawn as the recipe says.

    q, dO: [B, Hq, S, D]; k, v: [B, Hkv, S, D]. ``dO`` is None when
    ``with_do`` is False (it is still drawn last, so q/k/v never depend on it).
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn(B, Hq, S, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    dO = None
    if with_do:
        dO = (torch.randn(B, Hq, S, D, generator=g, dtype=torch.float32) * do_std).to(torch.bfloat16)
    return q, k, v, dO


def seq_bounds(lengths):
    """Bounds [0, l0, l0+l1, ...] of sequences laid end to end (int32 CPU tensor)."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def draw_lengths(n: int, lo: int, hi: int, seed: int):
    """n sequence lengths, uniform on [lo, hi], from their own seeded generator."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def make_packed_inputs(Hq: int, Hkv: int, lens_q, lens_k, D: int, seed: int,
                       do_std: float = 0.1, with_do: bool = True):
    """Packed batch: bf16 CPU tensors q [Hq, Tq, D], k, v [Hkv, Tk, D], dO [Hq, Tq, D] (or None)
    drawn in that order as the recipe says, plus the int32 bounds cu_q, cu_k."""
    cu_q = seq_bounds(lens_q)
    cu_k = seq_bounds(lens_k)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn(Hq, Tq, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(Hkv, Tk, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(Hkv, Tk, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    dO = None
    if with_do:
        dO = (torch.randn(Hq, Tq, D, generator=g, dtype=torch.float32) * do_std).to(torch.bfloat16)
    return q, k, v, dO, cu_q, cu_k


def rope_tables(S: int, D: int, base: float = 10000.0, offset: int = 0):
    """Rotary-position tables, the input a caller of the RoPE entry points supplies: f32 CPU
    tensors cos, sin of shape [S, D/2] with entry [p, i] = cos / sin((offset + p) * base**(-2i/D)),
    evaluated in float64 and rounded to float32."""
    i = torch.arange(D // 2, dtype=torch.float64)
    p = torch.arange(offset, offset + S, dtype=torch.float64)
    ang = p[:, None] * torch.pow(torch.tensor(float(base), dtype=torch.float64), -2.0 * i / D)[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


def workload_inputs(name: str, with_do: bool = True):
    w = WORKLOADS[name]
    return make_inputs(w.B, w.Hq, w.Hkv, w.S, w.D, w.seed, w.do_std, with_do)


def to_f64(t: torch.Tensor):
    """Exact widening of a bf16 tensor to a float64 numpy array (every bf16 value is an f64 value)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
