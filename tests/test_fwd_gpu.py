"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def run_fwd(inp):
    q, k, v = (parity.to_device(inp, n) for n in ("q", "k", "v"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, inp.causal, bm, kl)
    assert fa.fa_get_device_status() == 0
    return parity.to_host64(o), lse.cpu().numpy().astype(np.float64)


def oracle_fwd(inp, heads=None):
    return oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=inp.causal, kv_len=inp.kv_len,
                                    block_mask=inp.block_mask, heads=heads)


def test_tiny_fp32_workload():
    inp = inputs.workload_inputs("tiny_fp32")
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, fp32=True, what="tiny fp32")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 129, 200, 384])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_ragged_sizes(N, d, causal):
    inp = inputs.make_inputs(2, 3, N, d, seed=N * 7 + d + int(causal), causal=causal, with_dout=False)
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_jumps_between_key_tiles(d, causal):
    # Scores of even query rows jump between key tiles by a planted component (natural
    # log units 0, +5, +20, +28, -2 for key tiles 0..4), so the d = 128 kernel's three
    # per-tile paths all occur: exponentials against the running max kept (their sum at
    # most 2^8), the row max taken but the running max kept (within the rescale slack),
    # and the running max raised with an O rescale (+20, +28).  Odd rows keep plain
    # N(0,1)-scaled scores, so warps mix the cases.
    N = 640
    inp = inputs.make_inputs(1, 2, N, d, seed=901 + d + int(causal), causal=causal, with_dout=False)
    jump = np.array([0.0, 5.0, 20.0, 28.0, -2.0], np.float32)
    a = 8.0
    q, k = inp.q.copy(), inp.k.copy()
    q[:, :, 0::2, 0] = a
    q[:, :, 1::2, 0] = 0.0
    k[:, :, :, 0] = inputs.round_bf16(np.repeat(jump, 128)[None, None, :] * np.sqrt(d) / a)
    inp = dataclasses.replace(inp, q=q, k=k)
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, what=f"max jumps d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 77, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_ragged_sizes(N, d, causal):
    inp = inputs.make_inputs(1, 2, N, d, seed=N + d, dtype="fp32", causal=causal, with_dout=False)
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, fp32=True, what=f"fp32 N={N} d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_ragged(causal, d):
    inp = inputs.make_inputs(5, 2, 384, d, seed=31, causal=causal, kv_len_range=(1, 384), with_dout=False)
    inp.kv_len[:] = np.array([0, 1, 129, 200, 384], np.int32)  # 0: no key at all
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    parity.check_forward(o, lse, ro, rl, what="key padding")


@pytest.mark.parametrize("d", [64, 128])
def test_block_mask_with_empty_rows(d):
    inp = inputs.make_inputs(2, 2, 640, d, seed=41, with_dout=False,
                             block_mask=dict(band=1, global_cols=0, frac=0.2))
    inp.block_mask[2, :] = 0  # query tile 2 sees nothing: O = 0, LSE = -inf
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    assert np.all(o[:, :, 256:384] == 0) and np.all(np.isneginf(lse[:, :, 256:384]))
    parity.check_forward(o, lse, ro, rl, what="block mask")


def test_dense_block_mask_equals_no_mask_bitwise():
    inp = inputs.make_inputs(2, 2, 512, 128, seed=5, with_dout=False)
    o1, l1 = run_fwd(inp)
    inp.block_mask = np.ones((4, 4), np.uint8)
    o2, l2 = run_fwd(inp)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_causal_with_block_mask_and_padding(d):
    # at d = 128 the two query tiles of a CTA see different key tiles, so the two MMA
    # issuers walk key tiles that only one of them uses
    inp = inputs.make_inputs(2, 2, 700, d, seed=6, causal=True, kv_len_range=(300, 700), with_dout=False,
                             block_mask=dict(band=2, global_cols=1, frac=0.3))
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, what="causal+mask+padding")


def test_forward_is_deterministic():
    inp = inputs.make_inputs(1, 4, 1000, 128, seed=8, causal=True, with_dout=False)
    o1, l1 = run_fwd(inp)
    o2, l2 = run_fwd(inp)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_bert_large_padded_full_size():
    """Full BERT-large-shaped workload (B16 H16 N512 d64, key padding), every head."""
    inp = inputs.workload_inputs("bert_large_padded")
    o, lse = run_fwd(inp)
    ro, rl = oracle_fwd(inp)
    parity.check_forward(o, lse, ro, rl, what="bert")
