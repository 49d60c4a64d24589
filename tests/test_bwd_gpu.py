"""Backward parity: dQ, dK, dV from the CUDA path against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def run_fwd_bwd(inp):
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, inp.causal, bm, kl)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, inp.scale, inp.causal, bm, kl)
    assert fa.fa_get_device_status() == 0
    h = parity.to_host64
    return {"o": h(o), "lse": lse.cpu().numpy().astype(np.float64), "dq": h(dq), "dk": h(dk), "dv": h(dv)}


def oracle_bwd(inp, heads=None):
    return oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=inp.causal,
                                     kv_len=inp.kv_len, block_mask=inp.block_mask, heads=heads)


def check(inp, what):
    got = run_fwd_bwd(inp)
    ref = oracle_bwd(inp)
    parity.check_forward(got["o"], got["lse"], ref["o"], ref["lse"], what=what)
    return parity.check_grads(got, ref, what=what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 129, 200, 384])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_sizes(N, d, causal):
    inp = inputs.make_inputs(2, 2, N, d, seed=100 + N + d + int(causal), causal=causal)
    check(inp, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_zero_grads_for_padded_keys(causal, d):
    inp = inputs.make_inputs(5, 2, 384, d, seed=9, causal=causal, kv_len_range=(1, 384))
    inp.kv_len[:] = np.array([0, 1, 129, 200, 384], np.int32)  # 0: no key, so dQ = dK = dV = 0
    got = run_fwd_bwd(inp)
    ref = oracle_bwd(inp)
    parity.check_grads(got, ref, what="padding")
    for b, n in enumerate(inp.kv_len):
        assert np.all(got["dk"][b, :, n:] == 0) and np.all(got["dv"][b, :, n:] == 0)
    assert np.all(got["dq"][0] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_block_mask(d):
    inp = inputs.make_inputs(2, 2, 640, d, seed=12, block_mask=dict(band=1, global_cols=1, frac=0.2))
    inp.block_mask[3, :] = 0   # an empty query tile row
    inp.block_mask[:, 4] = 0   # a key tile no query sees: dK = dV = 0 there
    got = run_fwd_bwd(inp)
    ref = oracle_bwd(inp)
    parity.check_grads(got, ref, what="block mask")
    assert np.all(got["dq"][:, :, 384:512] == 0)
    assert np.all(got["dk"][:, :, 512:] == 0) and np.all(got["dv"][:, :, 512:] == 0)


def test_causal_block_mask_padding_d128():
    inp = inputs.make_inputs(2, 2, 520, 128, seed=13, causal=True, kv_len_range=(200, 520),
                             block_mask=dict(band=1, global_cols=1, frac=0.3))
    check(inp, "causal+mask+padding")


def test_bert_large_padded_full_size():
    """Full BERT-large-shaped workload (B16 H16 N512 d64, key padding), every head."""
    inp = inputs.workload_inputs("bert_large_padded")
    check(inp, "bert")


@pytest.mark.parametrize("d,N,causal", [(128, 4096, True), (128, 2048, False), (64, 4096, True)])
def test_long_whole_heads(d, N, causal):
    """Whole heads with many query tiles per key tile (32 at N = 4096), fwd + bwd
    element by element; dK, dV also key tile by key tile, so that one tile's error
    cannot hide in the whole-tensor norm."""
    inp = inputs.make_inputs(1, 2, N, d, seed=20 + d + N // 1024 + int(causal), causal=causal)
    got = run_fwd_bwd(inp)
    ref = oracle_bwd(inp)
    parity.check_forward(got["o"], got["lse"], ref["o"], ref["lse"], what=f"N={N} d={d}")
    parity.check_grads(got, ref, what=f"N={N} d={d}")
    for t in range(N // 128):
        sl = slice(t * 128, (t + 1) * 128)
        for name in ("dk", "dv", "dq"):
            e = parity.rel_fro(got[name][:, :, sl], ref[name][:, :, sl])
            assert e <= parity.GRAD_REL_FRO, f"N={N} d={d} tile {t} {name} rel-fro {e:.3g}"
