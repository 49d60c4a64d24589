"""Error model of the FP8 forward, for its parity tests.

The FP8 forward takes Q, K, V as E4M3 codes with one scale per tensor; the oracle
receives exactly the values those codes stand for, so input rounding is not an
error.  What remains is the kernel's own arithmetic:

  * P, the unnormalised probabilities exp(S - m) of one key tile, are rounded to
    E4M3 before the P V product (the tensor cores take both operands of one
    product in the same 8-bit family).  m is the row max the kernel uses at that
    tile, which lies at most 8 log2 units below the row max seen so far, so the
    rounded values lie in (0, 2^8].  A normal E4M3 value has 3 stored mantissa
    bits: round-to-nearest moves it by at most 2^-4 of itself; below 2^-6 the
    step is 2^-9, so the move is at most min(value, 2^-10).  Rescaling to the
    final row max multiplies value and error alike by a factor <= 1, hence per key
    |dP_ij| <= max(2^-4 P_ij, min(P_ij, 2^-10)) with P_ij = exp(S_ij - max_j S_ij).
  * The row sum l is taken over the unrounded values, so LSE = m + ln l is not
    touched by the rounding of P.
  * The score and output products accumulate on the tensor cores.  The bound
    allows each dot product a relative error of 2^-13 of the sum of absolute
    products (a narrower adder than fp32; fp32 gives far less).
  * O is rounded to bf16 (half an ulp is 2^-9 of |O|; the bound allows 2^-8).

fp8_forward_bounds() turns this into per-element bounds on |O - O_exact| and
|LSE - LSE_exact|.  The bound adds every rounding error with the same sign, so it
is loose by about the square root of the number of keys; the tight check is
statistical.  The relative error of round-to-nearest with 3 mantissa bits has an
RMS value below 2^-4 / sqrt(3) = 0.036.  O_i is a weighted sum of value rows with
independent zero-mean entries, so the Frobenius norm of the error relative to
the Frobenius norm of O has the same RMS.  The parity tests therefore ask for a
relative Frobenius error of at most 0.05 for O, and simulate_fp8_forward() (a CPU
model of the kernel's rounding of P, in fp64) is used to check both claims.
"""
from __future__ import annotations

import math

import numpy as np

from io_aware_exact_attention_gb300 import inputs

TILE = 128
O_REL_FRO_TOL = 0.05
ACC_REL = 2.0 ** -13   # allowance for the tensor-core adders, relative to the sum of |products|
SLACK_LOG2 = 8.0       # the kernel's row max may trail the running max by this much (log2 units)


def visible(N: int, causal: bool, kv_len: int | None, block_mask: np.ndarray | None,
            rows: np.ndarray) -> np.ndarray:
    """bool [len(rows), N]: which keys each query row sees (causal, key padding,
    128x128 tile mask)."""
    j = np.arange(N)[None, :]
    i = np.asarray(rows)[:, None]
    vis = np.ones((len(rows), N), bool)
    if causal:
        vis &= j <= i
    if kv_len is not None:
        vis &= j < min(max(int(kv_len), 0), N)
    if block_mask is not None:
        vis &= block_mask[i // TILE, j // TILE].astype(bool)
    return vis


def exact_rows(q, k, v, scale, vis):
    """fp64 S, P = exp(S - rowmax), l, O, LSE for one head's selected rows (q: [R, d])."""
    s = scale * (q.astype(np.float64) @ k.astype(np.float64).T)
    s = np.where(vis, s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.where(vis, np.exp(s - m_safe), 0.0)
    l = p.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l > 0, (p @ v.astype(np.float64)) / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[:, 0] > 0, m_safe[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return s, p, l, o, lse


def fp8_forward_bounds(q, k, v, scale, vis):
    """Per-element bounds (o_bound [R, d], lse_bound [R]) for one head's rows."""
    s, p, l, o, lse = exact_rows(q, k, v, scale, vis)
    absqk = scale * (np.abs(q.astype(np.float64)) @ np.abs(k.astype(np.float64)).T)
    ds = np.where(vis, ACC_REL * absqk + 2.0 ** -22 * np.abs(np.where(vis, s, 0.0)), 0.0)
    eta = np.expm1(2.0 * ds.max(axis=1, keepdims=True, initial=0.0))  # relative move of P and l
    dp = np.maximum(2.0 ** -4 * p, np.minimum(p, 2.0 ** -10)) * (1 + eta) + eta * p
    av = np.abs(v.astype(np.float64))
    l_safe = np.where(l > 0, l, 1.0)
    pv_abs = (p @ av) / l_safe
    o_bound = ((dp @ av) / l_safe + eta * np.abs(o)) / (1 - eta) + ACC_REL * pv_abs + 2.0 ** -8 * np.abs(o) + 1e-6
    lse_bound = ds.max(axis=1, initial=0.0) + 1e-5 * np.maximum(np.abs(np.where(np.isfinite(lse), lse, 0.0)), 1.0)
    return o_bound, lse_bound


def simulate_fp8_forward(q, k, v, scale, vis, tile=TILE, rng=None):
    """CPU model of the FP8 forward's treatment of P, in fp64: key tiles in order, a
    running max that is raised only when a tile's max exceeds it by more than 8
    log2 units, P' = 2^(log2e * S - m) rounded to E4M3 for the P V sum, unrounded P'
    for the row sum.  With `rng`, the max used at each tile is additionally lowered
    by a random amount in [0, 8) log2 units (within what the kernel may use), to
    exercise the whole range of P'.  Returns O [R, d] (fp64, not rounded to bf16)."""
    log2e = 1.0 / math.log(2.0)
    s = scale * (q.astype(np.float64) @ k.astype(np.float64).T) * log2e
    s = np.where(vis, s, -np.inf)
    R, N = s.shape
    o = np.zeros((R, v.shape[1]))
    l = np.zeros(R)
    m = np.full(R, -np.inf)
    seen = np.full(R, -np.inf)  # max over the keys so far
    v64 = v.astype(np.float64)
    for j0 in range(0, N, tile):
        st = s[:, j0:j0 + tile]
        mx = st.max(axis=1)
        seen = np.maximum(seen, mx)
        if rng is None:
            m_new = np.where(mx > m + SLACK_LOG2, mx, m)
        else:  # any non-decreasing max in [seen - 8, seen]
            m_new = np.maximum(m, seen - rng.uniform(0.0, SLACK_LOG2, size=R))
        m_use = np.where(np.isfinite(m_new), m_new, 0.0)
        alpha = np.where(np.isfinite(m), np.exp2(m - m_use), 0.0)
        pp = np.where(np.isfinite(st), np.exp2(st - m_use[:, None]), 0.0)
        pq = inputs.e4m3_bits_to_f32(inputs.e4m3_bits(pp.astype(np.float32))).astype(np.float64)
        # the float32 cast only trims digits far below E4M3's step
        l = l * alpha + pp.sum(axis=1)
        o = o * alpha[:, None] + pq @ v64[j0:j0 + tile]
        m = m_new
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)


def rel_fro(x, y) -> float:
    y = np.asarray(y, np.float64)
    n = float(np.linalg.norm(y))
    return float(np.linalg.norm(np.asarray(x, np.float64) - y) / n) if n > 0 else float(np.linalg.norm(x))
