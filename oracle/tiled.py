"""Blocked softmax attention in fp64 numpy, built from mergeable per-block states.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  It lets the tests check the
method's exactness claim independently of the CUDA path: a result assembled block
by block equals the materialised softmax result, for every way of cutting the
query and key axes into blocks (khetwal.com, "FlashAttention: how a memory trick
unlocked...", section "The Trick: Online Softmax"; the 128-row blocks of the
section "Tiling" and of the worked example's conceptual listing).

Formulation.  For one query row and any set J of its visible keys, the triple

    m_J = max_{j in J} s_j,   l_J = sum_{j in J} exp(s_j - m_J),
    a_J = sum_{j in J} exp(s_j - m_J) v_j

is all that is needed from J.  Two disjoint sets combine exactly:

    m = max(m_A, m_B),  w_A = exp(m_A - m),  w_B = exp(m_B - m),
    l = w_A l_A + w_B l_B,   a = w_A a_A + w_B a_B,

and after all keys O = a / l, LSE = m + ln l.  Folding the key blocks of a query
block into a running triple, left to right, is the online-softmax recurrence of
that section (running max, running normaliser, rescaled output).  Readings where
the pages are silent:
  * scores carry the scale factor (the score step of "The Quadratic Memory
    Bottleneck" applies a scale before the softmax);
  * the triple is kept per query row;
  * a block in which a row sees no key contributes the empty triple
    (m = -inf, l = 0, a = 0), whose weight in a merge is 0, so exp(-inf - -inf)
    is never formed;
  * a row that sees no key at all gets O = 0 and LSE = -inf.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def visible_mask(n, causal=False, kv_len=None, block_mask=None, tile=128):
    """Boolean [n, n] visibility: j < kv_len, j <= i if causal, tile bit set."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    vis = np.ones((n, n), dtype=bool)
    if kv_len is not None:
        vis &= j < int(kv_len)
    if causal:
        vis &= j <= i
    if block_mask is not None:
        bm = np.asarray(block_mask).astype(bool)
        vis &= bm[i // tile, j // tile]
    return vis


@dataclass
class RowState:
    """Per-row summary (m, l, a) of the keys seen so far, for a block of rows."""
    m: np.ndarray  # [rows] max score, -inf if no key
    l: np.ndarray  # [rows] sum of exp(score - m)
    a: np.ndarray  # [rows, d] sum of exp(score - m) * value row

    @staticmethod
    def empty(rows, d):
        return RowState(np.full(rows, -np.inf), np.zeros(rows), np.zeros((rows, d)))


def _weight(m_part, m_all):
    """exp(m_part - m_all), and 0 where the part is empty (m_part = -inf)."""
    out = np.zeros_like(m_part)
    has = np.isfinite(m_part)
    out[has] = np.exp(m_part[has] - m_all[has])
    return out


def block_state(scores, values, visible):
    """State of one key block: `scores` [rows, cols], `values` [cols, d], `visible` mask."""
    s = np.where(visible, scores, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    e = np.zeros_like(s)
    has = np.isfinite(m)
    e[has] = np.exp(s[has] - m[has, None])  # masked entries give exp(-inf) = 0
    return RowState(m, e.sum(axis=1), e @ values)


def merge(x: RowState, y: RowState) -> RowState:
    """Exact combination of the states of two disjoint key sets."""
    m = np.maximum(x.m, y.m)
    wx, wy = _weight(x.m, m), _weight(y.m, m)
    return RowState(m, wx * x.l + wy * y.l, wx[:, None] * x.a + wy[:, None] * y.a)


def finish(st: RowState):
    """(O, LSE) of a final state; rows with no key get O = 0, LSE = -inf."""
    seen = st.l > 0
    denom = np.where(seen, st.l, 1.0)
    o = np.where(seen[:, None], st.a / denom[:, None], 0.0)
    lse = np.where(seen, st.m + np.log(denom), -np.inf)
    return o, lse


def tiled_attention(q, k, v, scale, block_q, block_k, *, causal=False, kv_len=None,
                    block_mask=None, tile=128):
    """One head, q/k/v [N, d]; query blocks of `block_q` rows, key blocks of `block_k`.
    Returns (O [N, d], LSE [N]) in float64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape
    vis = visible_mask(n, causal, kv_len, block_mask, tile)
    o = np.zeros((n, d))
    lse = np.empty(n)
    for r0 in range(0, n, block_q):
        r1 = min(r0 + block_q, n)
        st = RowState.empty(r1 - r0, d)
        for c0 in range(0, n, block_k):
            c1 = min(c0 + block_k, n)
            part = block_state(scale * (q[r0:r1] @ k[c0:c1].T), v[c0:c1], vis[r0:r1, c0:c1])
            st = merge(st, part)
        o[r0:r1], lse[r0:r1] = finish(st)
    return o, lse
