"""Pins for the fp64 oracle: closed forms, invariants, finite differences and an
independent library routine.  None of these retypes the oracle's formula; each
is chosen so that a plausible slip in it (a dropped scale, a wrong sign or index,
a transposed operand, an off-by-one mask) fails at least one test here.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.tiled import tiled_attention, visible_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _eval(expr, symbols):
    env = {"sqrt": math.sqrt, "log": math.log, "__builtins__": {}}
    env.update(symbols)
    return float(eval(str(expr), env))  # fixture holds plain arithmetic only


def _head(q, k, v, dout, scale, **kw):
    r = oracle.head_rows(q, k, v, dout, scale, **kw)
    c = oracle.head_cols(q, k, v, dout, scale, r["m"], r["l"], r["D"], **kw)
    return r, c


# --------------------------------------------------------------- golden values

@pytest.mark.parametrize("variant", ["non_causal", "causal"])
def test_golden_hand_derived(variant):
    fx = json.load(open(os.path.join(GOLDEN, "tiny_closed_form.json")))
    sym = {}
    for name, expr in fx["symbols"].items():
        sym[name] = _eval(expr, sym)
    inp = {n: np.array([[_eval(x, sym) for x in row] for row in fx["inputs"][n]]) for n in ("q", "k", "v", "dout")}
    r, c = _head(inp["q"], inp["k"], inp["v"], inp["dout"], fx["inputs"]["scale"], causal=(variant == "causal"))
    exp = fx[variant]
    for name, got in (("o", r["o"]), ("dq", r["dq"]), ("dk", c["dk"]), ("dv", c["dv"])):
        want = np.array([[_eval(x, sym) for x in row] for row in exp[name]])
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14, err_msg=name)
    np.testing.assert_allclose(r["lse"], [_eval(x, sym) for x in exp["lse"]], rtol=1e-13)


# ------------------------------------------------------------------ invariants

def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("causal,kv_len,use_mask", [(False, None, False), (True, None, False),
                                                    (False, 19, False), (True, 23, True)])
def test_softmax_rows_sum_to_one(causal, kv_len, use_mask):
    # With V = identity (d = N) the output row is the probability row itself.
    rng = np.random.default_rng(1)
    n = 32
    q, k = 2.0 * _rand(rng, n, 8), _rand(rng, n, 8)
    q = np.concatenate([q, np.zeros((n, n - 8))], axis=1)
    k = np.concatenate([k, np.zeros((n, n - 8))], axis=1)
    v = np.eye(n)
    bm = None
    if use_mask:
        bm = np.array([[1, 0, 1, 1], [0, 1, 0, 1], [1, 1, 1, 0], [0, 0, 1, 1]], np.uint8)
    r = oracle.head_rows(q, k, v, None, 0.7, causal=causal, kv_len=kv_len, block_mask=bm, tile=8)
    p = r["o"]
    vis = visible_mask(n, causal, kv_len, bm, 8)
    rows = vis.any(axis=1)
    np.testing.assert_allclose(p[rows].sum(axis=1), 1.0, atol=1e-14)
    assert np.all(p >= 0)
    assert np.all(p[~vis] == 0)
    assert np.all(r["lse"][~rows] == -np.inf) and np.all(p[~rows] == 0)


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 11), (True, 11)])
def test_identical_keys_give_mean_of_values(causal, kv_len):
    rng = np.random.default_rng(2)
    n, d, scale = 24, 6, 0.37
    q, v = _rand(rng, n, d), _rand(rng, n, d)
    key = _rand(rng, d)
    k = np.tile(key, (n, 1))
    r = oracle.head_rows(q, k, v, None, scale, causal=causal, kv_len=kv_len)
    kl = n if kv_len is None else kv_len
    for i in range(n):
        count = min(i + 1, kl) if causal else kl
        np.testing.assert_allclose(r["o"][i], v[:count].mean(axis=0), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["lse"][i], scale * q[i] @ key + math.log(count), rtol=1e-13)


def test_dominant_score_selects_one_value_row():
    rng = np.random.default_rng(3)
    n, d, scale = 16, 16, 0.25
    k, _ = np.linalg.qr(_rand(rng, d, d))  # orthonormal key rows
    k = k[:n]
    v = _rand(rng, n, d)
    targets = rng.integers(0, n, size=n)
    c = 80.0 / scale  # score of the target key is 80, every other score 0
    q = c * k[targets]
    r = oracle.head_rows(q, k, v, None, scale)
    np.testing.assert_allclose(r["o"], v[targets], atol=1e-30 + 1e-12)
    np.testing.assert_allclose(r["lse"], 80.0 + np.log1p((n - 1) * np.exp(-80.0)), rtol=1e-14)


def test_single_key_and_causal_row_zero():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 1, 5), _rand(rng, 1, 5), _rand(rng, 1, 5)
    r = oracle.head_rows(q, k, v, None, 0.9)
    np.testing.assert_allclose(r["o"][0], v[0], rtol=1e-15)
    np.testing.assert_allclose(r["lse"][0], 0.9 * q[0] @ k[0], rtol=1e-14)
    q, k, v = _rand(rng, 9, 5), _rand(rng, 9, 5), _rand(rng, 9, 5)
    r = oracle.head_rows(q, k, v, None, 0.9, causal=True)
    np.testing.assert_allclose(r["o"][0], v[0], rtol=1e-15)
    np.testing.assert_allclose(r["lse"][0], 0.9 * q[0] @ k[0], rtol=1e-14)


def test_uniform_scores_give_mean():
    rng = np.random.default_rng(5)
    n, d = 20, 7
    k, v = _rand(rng, n, d), _rand(rng, n, d)
    r = oracle.head_rows(np.zeros((n, d)), k, v, None, 1.3, kv_len=13)
    np.testing.assert_allclose(r["o"], np.tile(v[:13].mean(0), (n, 1)), rtol=1e-13)
    np.testing.assert_allclose(r["lse"], math.log(13), rtol=1e-14)


def test_key_length_zero_and_truncation():
    """A key length L keeps keys [0, L): the result is attention over K[:L], V[:L]
    (written out with numpy here), and L = 0 leaves every row without a key: O = 0,
    LSE = -inf, dQ = 0 (fully masked rows); a length above N means no padding."""
    rng = np.random.default_rng(15)
    n, d = 12, 5
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    for L in (1, 7, n):
        r = oracle.head_rows(q, k, v, do, 0.6, kv_len=L)
        s = 0.6 * q @ k[:L].T
        p = np.exp(s - s.max(1, keepdims=True))
        np.testing.assert_allclose(r["o"], (p / p.sum(1, keepdims=True)) @ v[:L], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(r["lse"], s.max(1) + np.log(p.sum(1)), rtol=1e-14)
    r = oracle.head_rows(q, k, v, do, 0.6, kv_len=0)
    assert np.all(r["o"] == 0) and np.all(np.isneginf(r["lse"])) and np.all(r["dq"] == 0)
    full = oracle.head_rows(q, k, v, do, 0.6)
    np.testing.assert_array_equal(oracle.head_rows(q, k, v, do, 0.6, kv_len=n + 5)["o"], full["o"])
    out = oracle.attention_backward(q[None, None], k[None, None], v[None, None], do[None, None], 0.6,
                                    kv_len=np.array([0], np.int32))
    assert np.all(out["o"] == 0) and np.all(out["dk"] == 0) and np.all(out["dv"] == 0)


def test_permutation_equivariance():
    rng = np.random.default_rng(6)
    n, d = 30, 8
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    perm = rng.permutation(n)
    r1, c1 = _head(q, k, v, do, 0.4)
    r2, c2 = _head(q, k[perm], v[perm], do, 0.4)
    np.testing.assert_allclose(r1["o"], r2["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r1["lse"], r2["lse"], rtol=1e-13)
    np.testing.assert_allclose(r1["dq"], r2["dq"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(c1["dk"][perm], c2["dk"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(c1["dv"][perm], c2["dv"], rtol=1e-11, atol=1e-13)


def test_scale_enters_scores_only():
    # Scaling Q by t and the scale by 1/t leaves everything but dQ unchanged; dQ scales by 1/t.
    rng = np.random.default_rng(7)
    n, d, t = 17, 4, 2.5
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    r1, c1 = _head(q, k, v, do, 0.6, causal=True)
    r2, c2 = _head(q * t, k, v, do, 0.6 / t, causal=True)
    np.testing.assert_allclose(r1["o"], r2["o"], rtol=1e-12)
    np.testing.assert_allclose(r1["dq"], r2["dq"] * t, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(c1["dk"], c2["dk"], rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 21), (True, 9)])
def test_backward_sum_identities(causal, kv_len):
    # sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0, and sum_j dV_j = sum of dO over rows
    # that see at least one key -- properties that hold at any size.
    rng = np.random.default_rng(8)
    n, d = 40, 8
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    r, c = _head(q, k, v, do, 0.35, causal=causal, kv_len=kv_len)
    np.testing.assert_allclose(c["dk"].sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(c["dv"].sum(0), do.sum(0), rtol=1e-12, atol=1e-12)
    # rowwise: D_i = dO_i . O_i
    np.testing.assert_allclose(r["D"], np.einsum("ic,ic->i", do, r["o"]), rtol=1e-11, atol=1e-13)


# --------------------------------------------- exactness of the tiled algorithm

@pytest.mark.parametrize("causal,kv_len,use_mask", [(False, None, False), (True, None, False),
                                                    (False, 13, False), (True, 17, True)])
def test_tiled_equals_definition_for_every_block_split(causal, kv_len, use_mask):
    rng = np.random.default_rng(9)
    n, d = 20, 4
    q, k, v = 1.5 * _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]], np.uint8) if use_mask else None
    r = oracle.head_rows(q, k, v, None, 0.8, causal=causal, kv_len=kv_len, block_mask=bm, tile=8)
    for bq in range(1, n + 1):
        for bk in range(1, n + 1):
            o, lse = tiled_attention(q, k, v, 0.8, bq, bk, causal=causal, kv_len=kv_len, block_mask=bm, tile=8)
            np.testing.assert_allclose(o, r["o"], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse, r["lse"], rtol=1e-12, atol=1e-13)


def test_tiled_equals_definition_at_page_block_size():
    rng = np.random.default_rng(10)
    n, d = 300, 16
    q, k, v = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    r = oracle.head_rows(q, k, v, None, 0.25, causal=True)
    for bq, bk in ((128, 128), (64, 128), (128, 32), (100, 77)):
        o, lse = tiled_attention(q, k, v, 0.25, bq, bk, causal=True)
        np.testing.assert_allclose(o, r["o"], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse, r["lse"], rtol=1e-12)


def test_block_states_merge_in_any_order():
    # the merge of per-block states is exact, so folding the key blocks in reverse or
    # pairwise (tree) order gives the same state as the left-to-right fold, and the
    # empty state (no visible key) leaves a state unchanged
    from oracle.tiled import RowState, block_state, finish, merge
    rng = np.random.default_rng(11)
    n, d = 24, 5
    q, k, v = 2.0 * _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    vis = visible_mask(n, causal=True)
    parts = [block_state(0.7 * (q @ k[c:c + 5].T), v[c:c + 5], vis[:, c:c + 5]) for c in range(0, n, 5)]
    ref = oracle.head_rows(q, k, v, None, 0.7, causal=True)
    folds = []
    st = RowState.empty(n, d)
    for p in parts:
        st = merge(st, p)
    folds.append(st)
    st = RowState.empty(n, d)
    for p in reversed(parts):
        st = merge(p, st)
    folds.append(st)
    level = parts
    while len(level) > 1:
        level = [merge(level[i], level[i + 1]) if i + 1 < len(level) else level[i] for i in range(0, len(level), 2)]
    folds.append(merge(level[0], RowState.empty(n, d)))
    for st in folds:
        o, lse = finish(st)
        np.testing.assert_allclose(o, ref["o"], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, ref["lse"], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ finite differences

@pytest.mark.parametrize("causal,kv_len,use_mask", [(False, None, False), (True, None, False),
                                                    (False, 5, False), (True, 6, True)])
def test_gradients_match_central_differences(causal, kv_len, use_mask):
    rng = np.random.default_rng(11)
    n, d, scale, h = 8, 4, 0.7, 1e-6
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    bm = np.array([[1, 1], [0, 1]], np.uint8) if use_mask else None
    kw = dict(causal=causal, kv_len=kv_len, block_mask=bm, tile=4)
    r, c = _head(q, k, v, do, scale, **kw)

    def loss(qq, kk, vv):
        return float((oracle.head_rows(qq, kk, vv, None, scale, **kw)["o"] * do).sum())

    grads = {"q": r["dq"], "k": c["dk"], "v": c["dv"]}
    for name in ("q", "k", "v"):
        fd = np.zeros((n, d))
        for i in range(n):
            for j in range(d):
                args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                args[name][i, j] += h
                up = loss(args["q"], args["k"], args["v"])
                args[name][i, j] -= 2 * h
                dn = loss(args["q"], args["k"], args["v"])
                fd[i, j] = (up - dn) / (2 * h)
        err = np.abs(fd - grads[name]).max() / max(np.abs(grads[name]).max(), 1e-30)
        assert err < 1e-7, (name, err)


# ------------------------------------------------ independent library cross-check

@pytest.mark.parametrize("causal,use_len,use_mask", [(False, False, False), (True, False, False),
                                                     (False, True, False), (False, False, True),
                                                     (True, True, True)])
def test_against_torch_sdpa_fp64(causal, use_len, use_mask):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(12)
    B, H, n, d, tile = 2, 2, 96, 16, 32
    q, k, v, do = (rng.standard_normal((B, H, n, d)) for _ in range(4))
    kv_len = np.array([70, 96], np.int32) if use_len else None
    bm = None
    if use_mask:
        bm = (rng.random((n // tile, n // tile)) < 0.6).astype(np.uint8)
        bm[:, 0] = 1  # every query sees the first key tile, so no row is empty
    out = oracle.attention_backward(q, k, v, do, 0.3, causal=causal, kv_len=kv_len, block_mask=bm, tile=tile)
    # the torch side builds its boolean mask independently of the oracle
    allow = torch.ones(B, 1, n, n, dtype=torch.bool)
    ii = torch.arange(n)[:, None]
    jj = torch.arange(n)[None, :]
    if causal:
        allow &= (jj <= ii)
    if kv_len is not None:
        allow &= (jj[None, None] < torch.tensor(kv_len, dtype=torch.long)[:, None, None, None])
    if bm is not None:
        bmt = torch.tensor(bm, dtype=torch.bool)
        allow &= bmt[ii // tile, jj // tile]
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=allow, scale=0.3)
    o.backward(torch.tensor(do))
    s = 0.3 * tq.detach() @ tk.detach().transpose(-1, -2)
    lse = torch.logsumexp(s.masked_fill(~allow, -math.inf), dim=-1)
    np.testing.assert_allclose(out["o"], o.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["lse"], lse.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dq"], tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(out["dk"], tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(out["dv"], tv.grad.numpy(), rtol=1e-9, atol=1e-11)


# ------------------------------------------------------- sampled (subset) passes

def test_row_and_column_subsets_match_full_pass():
    rng = np.random.default_rng(13)
    n, d = 50, 8
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    r, c = _head(q, k, v, do, 0.5, causal=True)
    rows = np.array([49, 0, 17], np.int32)
    rs = oracle.head_rows(q, k, v, do, 0.5, causal=True, rows=rows)
    np.testing.assert_array_equal(rs["o"], r["o"][rows])
    np.testing.assert_array_equal(rs["dq"], r["dq"][rows])
    cols = np.array([3, 48], np.int32)
    cs = oracle.head_cols(q, k, v, do, 0.5, r["m"], r["l"], r["D"], causal=True, cols=cols)
    np.testing.assert_array_equal(cs["dk"], c["dk"][cols])
    np.testing.assert_array_equal(cs["dv"], c["dv"][cols])


def test_rejects_bad_arguments():
    z = np.zeros((4, 2))
    with pytest.raises(ValueError):
        oracle.head_rows(z, z, z, None, 1.0, rows=np.array([4], np.int32))
    with pytest.raises(ValueError):
        oracle.head_cols(z, z, z, z, 1.0, np.zeros(4), np.ones(4), np.zeros(4), cols=np.array([-1], np.int32))
