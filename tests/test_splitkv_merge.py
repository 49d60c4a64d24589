"""The split-KV merge rule, checked as an identity on the CPU (fp64).

A row's keys split into chunks; each chunk p gives O_p = sum_j exp(S_j - LSE_p) v_j with
LSE_p = log sum_j exp(S_j) over its keys (O_p = 0, LSE_p = -inf for a chunk without
keys).  Then LSE = log sum_p exp(LSE_p) and O = sum_p exp(LSE_p - LSE) O_p equal the
softmax over all keys.  The combine kernel applies exactly this rule to the partials
of the split-KV pass; these tests pin the rule itself."""
import numpy as np


def softmax_rows(s, v):
    m = s.max()
    p = np.exp(s - m)
    return p @ v / p.sum(), m + np.log(p.sum())


def partial(s, v):
    if s.size == 0:
        return np.zeros(v.shape[1]), -np.inf
    return softmax_rows(s, v)


def merge(parts):
    lses = np.array([lse for _, lse in parts])
    m = lses.max()
    if m == -np.inf:
        return np.zeros_like(parts[0][0]), -np.inf
    total = m + np.log(np.exp(lses - m).sum())
    return sum(np.exp(lse - total) * o for o, lse in parts), total


def test_merge_equals_full_softmax_for_any_chunking():
    rng = np.random.default_rng(0)
    for trial in range(200):
        n, d = int(rng.integers(1, 300)), 8
        s = rng.normal(0, 3, n)
        v = rng.normal(size=(n, d))
        cuts = np.sort(rng.integers(0, n + 1, size=int(rng.integers(0, 8))))
        bounds = [0, *cuts.tolist(), n]
        parts = [partial(s[a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]  # empty chunks included
        o, lse = merge(parts)
        o_ref, lse_ref = softmax_rows(s, v)
        np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


def test_merge_of_even_and_odd_tiles():
    # the partial pass gives each CTA's even and odd key tiles separate partials
    rng = np.random.default_rng(1)
    s = rng.normal(0, 2, 128 * 7 + 33)
    v = rng.normal(size=(s.size, 4))
    tiles = [np.arange(t * 128, min((t + 1) * 128, s.size)) for t in range((s.size + 127) // 128)]
    even = np.concatenate(tiles[0::2])
    odd = np.concatenate(tiles[1::2])
    o, lse = merge([partial(s[even], v[even]), partial(s[odd], v[odd])])
    o_ref, lse_ref = softmax_rows(s, v)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


def test_merge_of_no_keys_is_the_empty_row():
    o, lse = merge([partial(np.zeros(0), np.zeros((0, 3))) for _ in range(4)])
    assert np.all(o == 0) and lse == -np.inf
