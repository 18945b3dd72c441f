"""Oracle for causal grouped-query attention: plain, slow, f64, CPU.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import it. The product
path (the CUDA library and its Python binding) never imports, calls or links
anything here, and nothing here imports the product.

* ``oracle.attention`` -- forward (O, LSE) and backward (dQ, dK, dV) by the
  materialised definition, plus row-sampled variants of the same definition
  for workloads too large to evaluate whole.
* ``oracle.monoid``    -- the online-softmax (m, l, acc) monoid, used to pin
  the regrouping property the flash form rests on.
* ``oracle.decode``    -- a few new queries against a key/value cache
  (Sq <= Sk, bottom-right causal alignment).
* ``oracle.varlen``    -- variable-length sequences packed along the token
  axis (each sequence attends only to itself).
* ``oracle.rope``      -- rotary position embedding of Q and K before the
  attention (rotate-half pairing, caller-supplied cos/sin tables).

Pins (in ``tests/``): decimal brute force, central finite differences,
closed forms, invariants, torch f64 SDPA, monoid regrouping and a stored
golden file. Every function here is pinned; none is "parity unpinned".
"""

from . import attention, decode, monoid, rope, varlen  # noqa: F401
from .attention import (  # noqa: F401
    backward,
    backward_dkdv_rows,
    backward_dq_rows,
    forward,
    forward_rows,
    kv_head_of,
)
from .decode import forward_cached  # noqa: F401
from .rope import backward_rope, forward_rope  # noqa: F401
from .varlen import backward_varlen, forward_varlen  # noqa: F401
