"""The d = 64 kernels are persistent: a CTA walks several (query tile, head) items in
the forward and several (key tile, head) items in the backward.  These cases are
sized so that every CTA takes several items, with runs of batch entries whose key
length is 0 (every item of those heads has no visible key tile), mixed with
ordinary lengths, causal and not.

Exact checks on the empty heads (O = 0, LSE = -inf, dQ = dK = dV = 0), and the
fp64 oracle on a sample of the other heads within the usual tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_many_items_per_cta_with_empty_heads(causal):
    B, H, N, d = 40, 8, 384, 64  # 960 forward items over 304 CTAs, 960 backward items over 152 CTAs
    inp = inputs.make_inputs(B, H, N, d, seed=4242 + int(causal), causal=causal, kv_len_range=(1, N))
    pattern = [0, 0, 0, 384, 1, 0, 129, 0, 0, 200]  # consecutive empty batches, padding inside and across tiles
    inp.kv_len[:] = np.array([pattern[b % len(pattern)] for b in range(B)], np.int32)
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, causal, bm, kl)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, inp.scale, causal, bm, kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0

    empty = [b for b in range(B) if inp.kv_len[b] == 0]
    full = [b for b in range(B) if inp.kv_len[b] > 0]
    e = torch.tensor(empty, device="cuda")
    assert torch.count_nonzero(o.index_select(0, e)) == 0
    assert bool(torch.all(lse.index_select(0, e) == float("-inf")))
    for t in (dq, dk, dv):
        assert torch.count_nonzero(t.index_select(0, e)) == 0
    # padded keys of the other heads get no gradient
    for b in full:
        n = int(inp.kv_len[b])
        assert torch.count_nonzero(dk[b, :, n:]) == 0 and torch.count_nonzero(dv[b, :, n:]) == 0

    heads = [(full[0], 0), (full[1], 7), (full[2], 3), (full[-1], 5)]
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=causal, kv_len=inp.kv_len,
                                    heads=heads)
    h = parity.to_host64
    for b, hh in heads:
        got = {"o": h(o[b, hh]), "dq": h(dq[b, hh]), "dk": h(dk[b, hh]), "dv": h(dv[b, hh])}
        parity.check_forward(got["o"], lse[b, hh].cpu().numpy().astype(np.float64), ref["o"][b, hh],
                             ref["lse"][b, hh], what=f"head {b},{hh}")
        parity.check_grads(got, {n: ref[n][b, hh] for n in ("dq", "dk", "dv")}, what=f"head {b},{hh}")


@pytest.mark.parametrize("causal", [False, True])
def test_many_items_per_cta_block_mask_with_empty_rows_and_columns(causal):
    B, H, N, d = 16, 8, 1024, 64  # 1024 items in each direction, several per persistent CTA
    inp = inputs.make_inputs(B, H, N, d, seed=5151 + int(causal), causal=causal,
                             block_mask=dict(band=1, global_cols=0, frac=0.15))
    T = N // 128
    inp.block_mask[2, :] = 0      # query tile 2 sees nothing: O = 0, LSE = -inf on its rows
    inp.block_mask[5, :] = 0
    inp.block_mask[:, 6] = 0      # key tile 6 is seen by no query: dK = dV = 0 on its rows
    inp.block_mask[:, 3] = 0
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, causal, bm, kl)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, inp.scale, causal, bm, kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0

    for qt in (2, 5):
        rows = slice(qt * 128, (qt + 1) * 128)
        assert torch.count_nonzero(o[:, :, rows]) == 0
        assert bool(torch.all(lse[:, :, rows] == float("-inf")))
        assert torch.count_nonzero(dq[:, :, rows]) == 0
    for kt in (3, 6):
        rows = slice(kt * 128, (kt + 1) * 128)
        assert torch.count_nonzero(dk[:, :, rows]) == 0 and torch.count_nonzero(dv[:, :, rows]) == 0

    heads = [(0, 0), (5, 3), (11, 6), (15, 7)]
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=causal,
                                    block_mask=inp.block_mask, heads=heads)
    h = parity.to_host64
    for b, hh in heads:
        got = {"o": h(o[b, hh]), "dq": h(dq[b, hh]), "dk": h(dk[b, hh]), "dv": h(dv[b, hh])}
        parity.check_forward(got["o"], lse[b, hh].cpu().numpy().astype(np.float64), ref["o"][b, hh],
                             ref["lse"][b, hh], what=f"head {b},{hh}")
        parity.check_grads(got, {n: ref[n][b, hh] for n in ("dq", "dk", "dv")}, what=f"head {b},{hh}")
    assert T == 8
