"""Oracle: the online-softmax monoid in f64 (the derived, streaming form of one attention row).

TEST INFRASTRUCTURE, like the rest of ``oracle/``.

tang, "How tang works" section 3: the ``stabilize_softmax`` rewrite turns the
row max and the two sums of attention into one reduction whose state is
updated per key; "three running values carry everything needed", and the
combine "is associative, so it tiles and parallelizes like any sum".
Equation (6) itself is missing from the extracted text, so the state and the
combine below are the plainest reading of that prose:

  state of a set of keys J for one query row: (m, l, a) with
      m = max_{j in J} s_j,
      l = sum_{j in J} exp(s_j - m),
      a = sum_{j in J} exp(s_j - m) v_j          (a vector of length D);
  combine (m, l, a) + (m', l', a') = (M, l e^{m-M} + l' e^{m'-M}, a e^{m-M} + a' e^{m'-M}),
      M = max(m, m');
  identity (-inf, 0, 0); result O = a / l, LSE = m + ln l.

A state may also carry a *reference* value r >= m in place of m (the lazy
rescale the CUDA kernels use): (r, sum exp(s_j - r), sum exp(s_j - r) v_j)
describes the same set of keys, and a / l and r + ln l are unchanged.
"""

from __future__ import annotations

import numpy as np

IDENTITY_M = -np.inf


def identity(D: int):
    return (IDENTITY_M, 0.0, np.zeros(D))


def leaf(s_j: float, v_j):
    """State of the single key j: (s_j, 1, v_j)."""
    return (float(s_j), 1.0, np.asarray(v_j, dtype=np.float64).copy())


def _rescale(m_from: float, m_to: float) -> float:
    # exp(m_from - m_to), with the identity's -inf giving 0 and -inf - -inf avoided.
    if m_from == -np.inf:
        return 0.0
    return float(np.exp(m_from - m_to))


def combine(x, y):
    """The associative combine of two states."""
    m1, l1, a1 = x
    m2, l2, a2 = y
    M = max(m1, m2)
    if M == -np.inf:
        return (M, 0.0, np.zeros_like(a1))
    c1 = _rescale(m1, M)
    c2 = _rescale(m2, M)
    return (M, l1 * c1 + l2 * c2, a1 * c1 + a2 * c2)


def chunk_state(s, V):
    """State of a chunk of keys from its scores s [n] and values V [n, D], by the definition."""
    s = np.asarray(s, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if s.size == 0 or np.all(s == -np.inf):
        return identity(V.shape[1])
    m = float(s.max())
    w = np.exp(s - m)
    return (m, float(w.sum()), w @ V)


def with_reference(state, r: float):
    """The same state re-expressed against a reference r >= m."""
    m, l, a = state
    if m == -np.inf:
        return (r, 0.0, a * 0.0)
    c = float(np.exp(m - r))
    return (r, l * c, a * c)


def finish(state):
    """(O, LSE) of a state: O = a / l, LSE = m + ln l."""
    m, l, a = state
    return a / l, m + np.log(l)


def fold_left(states):
    acc = identity(states[0][2].shape[0]) if states else None
    for st in states:
        acc = combine(acc, st)
    return acc


def fold_tree(states):
    """Pairwise (balanced-tree) reduction of a list of states."""
    cur = list(states)
    while len(cur) > 1:
        nxt = [combine(cur[i], cur[i + 1]) for i in range(0, len(cur) - 1, 2)]
        if len(cur) % 2:
            nxt.append(cur[-1])
        cur = nxt
    return cur[0]


def stream_row(s, V, chunk_bounds):
    """Online softmax of one row, streaming the keys in chunks [b_0:b_1), [b_1:b_2), ...

    Returns the left fold of the chunk states (the order a single pass over
    the keys would use).
    """
    states = [chunk_state(s[a:b], V[a:b]) for a, b in zip(chunk_bounds[:-1], chunk_bounds[1:])]
    return fold_left(states)
