"""Parity at the full sizes of the five workloads, in the launch configuration the
benchmark times (one fa_fwd and one fa_bwd over the whole batch).

Where the fp64 oracle cannot redo the whole workload in seconds it checks what it
can compute one row or one column at a time:
  * whole heads, element by element (O, LSE, dQ, dK, dV), where one head takes the
    oracle seconds: GPT-2, block-sparse, and one 16k causal head (whose first key
    tile accumulates over all 128 query tiles);
  * at 64k, every query row of the last quarter of one head (O, LSE, dQ) and the dK,
    dV of three key tiles whose query rows all lie in that quarter (up to 128 query
    tiles accumulated per key tile), plus sampled rows of other heads;
and, on every head, identities that hold at any size:
  sum_j dK_j = 0 and sum_j dV_j = sum of dO over rows that see a key.
"""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def run_workload(inp):
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, inp.causal, bm, kl)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, inp.scale, inp.causal, bm, kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv, do=do)


def h64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_rows(inp, out, heads, rows):
    """O, LSE and dQ of the given query rows of the given heads against the oracle."""
    got = {n: [] for n in ("o", "lse", "dq")}
    ref = {n: [] for n in ("o", "lse", "dq")}
    rows = np.asarray(rows, np.int32)
    for b, h in heads:
        kl = None if inp.kv_len is None else int(inp.kv_len[b])
        r = oracle.head_rows(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.dout[b, h], inp.scale, causal=inp.causal,
                             kv_len=kl, block_mask=inp.block_mask, rows=rows)
        idx = torch.from_numpy(rows.astype(np.int64)).cuda()
        got["o"].append(h64(out["o"][b, h].index_select(0, idx)))
        got["lse"].append(out["lse"][b, h].index_select(0, idx).cpu().numpy().astype(np.float64))
        got["dq"].append(h64(out["dq"][b, h].index_select(0, idx)))
        ref["o"].append(r["o"])
        ref["lse"].append(r["lse"])
        ref["dq"].append(r["dq"])
    g = {n: np.stack(v) for n, v in got.items()}
    f = {n: np.stack(v) for n, v in ref.items()}
    parity.check_forward(g["o"], g["lse"], f["o"], f["lse"], what="sampled rows")
    e = parity.rel_fro(g["dq"], f["dq"])
    assert e <= parity.GRAD_REL_FRO, f"sampled dq rel-fro {e:.3g}"


def check_last_key_tile(inp, out, head):
    """dK, dV of every key in the last tile of a causal head (seen only by the last rows)."""
    b, h = head
    N = inp.q.shape[2]
    j0 = ((N - 1) // 128) * 128
    rows = np.arange(j0, N, dtype=np.int32)
    r = oracle.head_rows(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.dout[b, h], inp.scale, causal=True, rows=rows)
    m, l, D = (np.full(N, np.nan) for _ in range(3))
    m[rows], l[rows], D[rows] = r["m"], r["l"], r["D"]
    c = oracle.head_cols(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.dout[b, h], inp.scale, m, l, D, causal=True,
                         cols=rows)
    for name in ("dk", "dv"):
        got = h64(out[name][b, h, j0:N])
        e = parity.rel_fro(got, c[name])
        assert e <= parity.GRAD_REL_FRO, f"last key tile {name} rel-fro {e:.3g}"


def check_causal_head_block(inp, out, head, row0, key_tiles):
    """Causal head: O, LSE, dQ of every query row in [row0, N) and dK, dV of the given
    key tiles (each at or after row0, so every query that sees them is in the block),
    element by element against the oracle."""
    b, h = head
    N = inp.q.shape[2]
    rows = np.arange(row0, N, dtype=np.int32)
    r = oracle.head_rows(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.dout[b, h], inp.scale, causal=True, rows=rows)
    lse = out["lse"][b, h, row0:].cpu().numpy().astype(np.float64)
    parity.check_forward(h64(out["o"][b, h, row0:]), lse, r["o"], r["lse"], what=f"head {b},{h} rows {row0}..")
    e = parity.rel_fro(h64(out["dq"][b, h, row0:]), r["dq"])
    assert e <= parity.GRAD_REL_FRO, f"head {b},{h} rows {row0}.. dq rel-fro {e:.3g}"
    m, l, D = (np.full(N, np.nan) for _ in range(3))
    m[rows], l[rows], D[rows] = r["m"], r["l"], r["D"]
    cols = np.concatenate([np.arange(t * 128, min(N, t * 128 + 128)) for t in key_tiles]).astype(np.int32)
    assert cols.min() >= row0
    c = oracle.head_cols(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.dout[b, h], inp.scale, m, l, D, causal=True,
                         cols=cols)
    idx = torch.from_numpy(cols.astype(np.int64)).cuda()
    for name in ("dk", "dv"):
        got = h64(out[name][b, h].index_select(0, idx))
        e = parity.rel_fro(got, c[name])
        assert e <= parity.GRAD_REL_FRO, f"head {b},{h} key tiles {key_tiles} {name} rel-fro {e:.3g}"
        for t in range(len(key_tiles)):  # each tile on its own as well
            sl = slice(t * 128, (t + 1) * 128)
            e = parity.rel_fro(got[sl], c[name][sl])
            assert e <= parity.GRAD_REL_FRO, f"head {b},{h} key tile {key_tiles[t]} {name} rel-fro {e:.3g}"


def check_identities(inp, out):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (rows that see a key) on every head, in fp64."""
    f64 = torch.float64
    dk_sum = out["dk"].sum(dim=2, dtype=f64)
    dv_sum = out["dv"].sum(dim=2, dtype=f64)
    do_sum = out["do"].sum(dim=2, dtype=f64)
    dk_scale = out["dk"].abs().sum(dim=2, dtype=f64)
    dv_scale = out["dv"].abs().sum(dim=2, dtype=f64)
    # bf16 outputs: each term carries relative error <= 2^-9; the sums of N terms stay well inside 1e-2 of sum |x|
    assert float((dk_sum.abs() / dk_scale.clamp_min(1e-30)).max()) < 1e-2
    assert float(((dv_sum - do_sum).abs() / dv_scale.clamp_min(1e-30)).max()) < 1e-2


def test_gpt2_causal_full_size():
    inp = inputs.workload_inputs("gpt2_causal")
    out = run_workload(inp)
    heads = [(0, 0), (3, 7), (7, 11)]
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=True, heads=heads)
    for b, h in heads:
        got = {n: h64(out[n][b, h]) for n in ("o", "dq", "dk", "dv")}
        lse = out["lse"][b, h].cpu().numpy().astype(np.float64)
        parity.check_forward(got["o"], lse, ref["o"][b, h], ref["lse"][b, h], what=f"gpt2 head {b},{h}")
        parity.check_grads(got, {n: ref[n][b, h] for n in ("dq", "dk", "dv")}, what=f"gpt2 head {b},{h}")
    check_identities(inp, out)


def test_long_causal_16k_full_size():
    inp = inputs.workload_inputs("long_causal_16k")
    out = run_workload(inp)
    N = inp.q.shape[2]
    # one whole head, element by element, every key tile also on its own: key tile 0
    # is seen by all 128 query tiles
    check_causal_head_block(inp, out, (0, 5), 0, list(range(N // 128)))
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 8191, N - 1], rng.integers(0, N, 40)]))
    check_rows(inp, out, [(0, 0), (0, 13), (0, 31)], rows)
    check_last_key_tile(inp, out, (0, 5))
    check_identities(inp, out)


def test_long_causal_64k_full_size_and_linear_memory():
    inp = inputs.workload_inputs("long_causal_64k")
    free_before = torch.cuda.mem_get_info()[0]
    out = run_workload(inp)
    used = free_before - torch.cuda.mem_get_info()[0]
    N = inp.q.shape[2]
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 2, 65535, 32768], rng.integers(0, N, 12)]))
    check_rows(inp, out, [(0, 0), (0, 20)], rows)
    check_last_key_tile(inp, out, (0, 9))
    # the last quarter of one head: key tile 384 accumulates over 128 query tiles
    check_causal_head_block(inp, out, (0, 9), 3 * N // 4, [384, 448, 511])
    check_identities(inp, out)
    # memory is linear in N: the library allocates nothing, and the caller-side
    # buffers are the [B,H,N,d] tensors plus the O(B*H*N*d) workspace -- far from
    # the N x N fp32 score matrix (65536^2 * 4 B = 17 GB per head, 550 GB for 32 heads)
    B, H, _, d = inp.q.shape
    ws = fa.fa_bwd_workspace_size(B, H, N, d)
    assert ws == (B * H * N * 4 + 255) // 256 * 256 + (B * H * N * d * 4 + 255) // 256 * 256
    assert ws < 0.01 * (N * N * 4 * B * H)
    tensor_bytes = 9 * B * H * N * d * 2 + B * H * N * 4
    assert used < tensor_bytes + ws + (1 << 30), (used, tensor_bytes, ws)


def test_block_sparse_8k_full_size():
    inp = inputs.workload_inputs("block_sparse_8k")
    out = run_workload(inp)
    heads = [(0, 0), (3, 15)]
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, block_mask=inp.block_mask, heads=heads)
    for b, h in heads:
        got = {n: h64(out[n][b, h]) for n in ("o", "dq", "dk", "dv")}
        lse = out["lse"][b, h].cpu().numpy().astype(np.float64)
        parity.check_forward(got["o"], lse, ref["o"][b, h], ref["lse"][b, h], what=f"sparse head {b},{h}")
        parity.check_grads(got, {n: ref[n][b, h] for n in ("dq", "dk", "dv")}, what=f"sparse head {b},{h}")
    check_identities(inp, out)


def test_bert_large_padded_identities():
    inp = inputs.workload_inputs("bert_large_padded")
    out = run_workload(inp)
    # padded keys get exactly zero gradients
    for b, n in enumerate(inp.kv_len):
        assert torch.count_nonzero(out["dk"][b, :, n:]) == 0 and torch.count_nonzero(out["dv"][b, :, n:]) == 0
    check_identities(inp, out)
