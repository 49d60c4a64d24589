"""Parity of the split-KV forward (fa_fwd_splitkv) with the fp64 oracle.

The oracle takes one sequence length for queries and keys; for this non-causal
operation the query block or the keys are zero-padded to a common length, the padded
keys masked by the key length, which leaves every real row's result unchanged."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def dev(inp, name):
    return torch.from_numpy(inp.device_array(name).view(np.int16)).view(torch.bfloat16).cuda()


def run(inp, n_splits):
    q, k, v = dev(inp, "q"), dev(inp, "k"), dev(inp, "v")
    kl = torch.from_numpy(inp.kv_len).cuda() if inp.kv_len is not None else None
    o, lse = fa.attention_forward_splitkv(q, k, v, inp.scale, kl, n_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return parity.to_host64(o), lse.cpu().numpy().astype(np.float64)


def oracle_rows(inp, b, h, rows):
    Nq, d = inp.q.shape[2:]
    Nk = inp.k.shape[2]
    n = max(Nq, Nk)
    q = np.zeros((n, d), np.float32)
    k = np.zeros((n, d), np.float32)
    v = np.zeros((n, d), np.float32)
    q[:Nq], k[:Nk], v[:Nk] = inp.q[b, h], inp.k[b, h], inp.v[b, h]
    kl = Nk if inp.kv_len is None else min(max(int(inp.kv_len[b]), 0), Nk)
    r = oracle.head_rows(q, k, v, None, inp.scale, kv_len=kl, rows=np.asarray(rows, np.int32))
    return r["o"], r["lse"]


def check(inp, o, lse, heads=None, rows=None):
    B, H, Nq, _ = inp.q.shape
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    rows = np.arange(Nq) if rows is None else np.asarray(rows)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b, h in heads:
        ro, rl = oracle_rows(inp, b, h, rows)
        got_o.append(o[b, h][rows])
        got_l.append(lse[b, h][rows])
        ref_o.append(ro)
        ref_l.append(rl)
    parity.check_forward(np.stack(got_o), np.stack(got_l), np.stack(ref_o), np.stack(ref_l), what="split-KV")


@pytest.mark.parametrize("B,H,Nq,Nk,n_splits,kv", [
    (2, 4, 1, 5000, None, None),            # decode, automatic split count
    (2, 3, 77, 3000, 3, [0, 1777]),         # key padding, one sequence without keys
    (1, 2, 300, 1000, 1, None),             # three query tiles, one chunk
    (1, 2, 128, 4096, 16, None),            # many chunks of two key tiles
    (1, 1, 200, 130, 7, None),              # more chunks than key tiles, Nq > Nk
    (1, 2, 64, 129, 1, None),               # a chunk whose odd slot sees one ragged tile
])
def test_splitkv_matches_oracle(B, H, Nq, Nk, n_splits, kv):
    inp = inputs.make_qk_inputs(B, H, Nq, Nk, 128, seed=Nq + Nk)
    if kv is not None:
        inp.kv_len = np.array(kv, np.int32)
    o, lse = run(inp, n_splits)
    check(inp, o, lse)
    if kv is not None:
        empty = [b for b, n in enumerate(kv) if n == 0]
        for b in empty:
            assert np.all(o[b] == 0) and np.all(np.isneginf(lse[b]))


@pytest.mark.parametrize("n_splits", [1, 2])
def test_splitkv_running_max_jumps_between_key_tiles(n_splits):
    # Even query rows get a planted score component that jumps between key tiles
    # (natural log units 0, +5, +20, +28, -2 for key tiles 0..4).  A partial pass
    # hands even and odd key tiles to its two query slots, so each slot's running max
    # jumps too (0, +20, -2 and +5, +28) and the fast exponentials, the kept offset
    # and the O rescale all occur, with or without a key split.
    Nq, Nk, d = 256, 640, 128
    inp = inputs.make_qk_inputs(1, 2, Nq, Nk, d, seed=961 + n_splits)
    jump = np.array([0.0, 5.0, 20.0, 28.0, -2.0], np.float32)
    a = 8.0
    q, k = inp.q.copy(), inp.k.copy()
    q[:, :, 0::2, 0] = a
    q[:, :, 1::2, 0] = 0.0
    k[:, :, :, 0] = inputs.round_bf16(np.repeat(jump, 128)[None, None, :] * np.float32(np.sqrt(d) / a))
    inp = dataclasses.replace(inp, q=q, k=k)
    o, lse = run(inp, n_splits)
    check(inp, o, lse)


def test_splitkv_no_keys():
    inp = inputs.make_qk_inputs(1, 2, 50, 0, 128, seed=3)
    q = dev(inp, "q")
    k = torch.empty((1, 2, 0, 128), device="cuda", dtype=torch.bfloat16)
    o, lse = fa.attention_forward_splitkv(q, k, k, inp.scale, None, 2)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_splitkv_split_count_changes_rounding_only():
    inp = inputs.make_qk_inputs(1, 2, 128, 2048, 128, seed=5)
    o1, l1 = run(inp, 1)
    o8, l8 = run(inp, 8)
    assert np.max(np.abs(o1 - o8)) <= 2 ** -7 * np.max(np.abs(o1)) and np.max(np.abs(l1 - l8)) <= 1e-5


@pytest.mark.parametrize("name", sorted(inputs.QK_WORKLOADS))
def test_splitkv_workloads_sampled(name):
    """Full workload shapes in the launch configuration the bench times (automatic split
    count); sampled heads and rows against the oracle."""
    inp = inputs.qk_workload_inputs(name)
    o, lse = run(inp, None)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    B, H, Nq, _ = inp.q.shape
    rng = np.random.default_rng(11)
    heads = [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(3)]
    rows = np.unique(np.concatenate([[0, Nq - 1], rng.integers(0, Nq, 16)]))
    check(inp, o, lse, heads=heads, rows=rows)


def test_splitkv_decode_beyond_l2():
    """Decode of one query row against 16384 keys for B2 H32 (K, V 268 MB, twice the
    129 MB L2), automatic split count; sampled heads against the oracle."""
    inp = inputs.make_qk_inputs(2, 32, 1, 16384, 128, seed=12)
    o, lse = run(inp, None)
    check(inp, o, lse, heads=[(0, 0), (1, 17), (1, 31)])
