"""FP8 inputs and the FP8 forward's error model, checked on the CPU.

The E4M3 codec is pinned to PyTorch's float8_e4m3fn conversion (an independent
library routine); the error model is pinned by a worst case it must cover and
nearly reach, by the CPU simulation of the kernel's rounding of P staying inside
it, and by a planted packing mistake that the statistical tolerance must catch.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from io_aware_exact_attention_gb300 import inputs
from tests import fp8_error_model as M


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = inputs.e4m3_bits_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-16, 9, 200_000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(inputs.e4m3_bits(x), ref)


def test_e4m3_ties_round_to_even_and_range_edges():
    pos = inputs.e4m3_bits_to_f32(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in float32
    codes = inputs.e4m3_bits(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    assert np.array_equal(codes, np.where(lo % 2 == 0, lo, lo + 1))
    assert np.array_equal(inputs.e4m3_bits(-mids), codes | 0x80)
    assert inputs.e4m3_bits(np.float32([455.9]))[0] == 0x7E
    assert inputs.e4m3_bits(np.float32([2.0 ** -11]))[0] == 0  # half the subnormal step: ties to 0
    with pytest.raises(ValueError):
        inputs.e4m3_bits(np.float32([470.0]))
    with pytest.raises(ValueError):
        inputs.e4m3_bits(np.float32([np.nan]))


def test_quantize_uses_smallest_power_of_two_scale():
    x = np.random.default_rng(3).standard_normal((4, 300)).astype(np.float32)
    codes, s, xq = inputs.quantize_e4m3(x)
    assert math.log2(s) == int(math.log2(s))
    amax = np.abs(x).max()
    assert amax / s <= 448 < amax / (s / 2)
    assert np.array_equal(xq, inputs.e4m3_bits_to_f32(codes) * np.float32(s))
    rel = np.abs(xq - x) / np.maximum(np.abs(x), 2.0 ** -6 * s)
    assert rel.max() <= 2.0 ** -4 + 1e-7


def test_fp8_inputs_layout():
    inp = inputs.make_fp8_inputs(2, 3, 200, 128, seed=9, causal=True, kv_len_range=(50, 200))
    assert inp.ldv % 16 == 0 and inp.ldv >= 200
    assert inp.vt8.shape == (2, 3, 128, inp.ldv)
    assert np.array_equal(inp.vt8[..., :200], np.swapaxes(inputs.e4m3_bits(inp.v / np.float32(inp.descale_v)), 2, 3))
    assert not inp.vt8[..., 200:].any()
    assert np.array_equal(inp.q, inputs.e4m3_bits_to_f32(inp.q8) * np.float32(inp.descale_q))
    raw = inputs.make_inputs(2, 3, 200, 128, seed=9, dtype="fp32", causal=True, kv_len_range=(50, 200))
    assert np.array_equal(inp.kv_len, raw.kv_len)
    assert np.abs(inp.k - raw.k).max() <= 2.0 ** -4 * np.abs(raw.k).max()


def test_fp8_inputs_from_quantizes_given_draws():
    # the helper behind make_fp8_inputs: the same result from the same fp32 draws, and
    # planted values (as the FP8 running-max tests use) quantized like the rest
    raw = inputs.make_inputs(1, 2, 300, 128, seed=11, dtype="fp32", causal=True, with_dout=False)
    a = inputs.make_fp8_inputs(1, 2, 300, 128, seed=11, causal=True)
    b = inputs.fp8_inputs_from(raw)
    for name in ("q8", "k8", "vt8", "q", "k", "v"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    assert (a.descale_q, a.descale_k, a.descale_v, a.ldv, a.causal) == (b.descale_q, b.descale_k, b.descale_v, b.ldv,
                                                                       b.causal)
    k = raw.k.copy()
    k[..., 0] = 40.0
    c = inputs.fp8_inputs_from(dataclasses.replace(raw, k=k))
    assert c.descale_k > b.descale_k  # the larger planted column sets the tensor's scale
    assert np.array_equal(c.k, inputs.e4m3_bits_to_f32(c.k8) * np.float32(c.descale_k))
    assert np.all(c.k[..., 0] == 40.0)  # 40 = 320 * 2^-3 is exact in E4M3


def _head(inp, b, h, rows=None):
    N = inp.q.shape[2]
    rows = np.arange(N) if rows is None else rows
    kv = None if inp.kv_len is None else int(inp.kv_len[b])
    vis = M.visible(N, inp.causal, kv, inp.block_mask, rows)
    return inp.q[b, h][rows], inp.k[b, h], inp.v[b, h], vis


@pytest.mark.parametrize("case", ["causal", "padded", "blocks"])
def test_simulated_rounding_stays_inside_the_bound(case):
    if case == "causal":
        inp = inputs.make_fp8_inputs(1, 1, 600, 128, seed=21, causal=True)
    elif case == "padded":
        inp = inputs.make_fp8_inputs(2, 1, 520, 128, seed=22, kv_len_range=(130, 400))
    else:
        inp = inputs.make_fp8_inputs(1, 1, 768, 128, seed=23, block_mask=dict(band=1, global_cols=1, frac=0.2))
    rng = np.random.default_rng(5)
    for b in range(inp.q.shape[0]):
        q, k, v, vis = _head(inp, b, 0)
        ob, lb = M.fp8_forward_bounds(q, k, v, inp.scale, vis)
        o = M.exact_rows(q, k, v, inp.scale, vis)[3]
        for r in (None, rng):
            osim = M.simulate_fp8_forward(q, k, v, inp.scale, vis, rng=r)
            assert np.all(np.abs(osim - o) <= ob)
            assert 0.005 < M.rel_fro(osim, o) <= M.O_REL_FRO_TOL


def test_bound_is_reached_by_aligned_rounding_errors():
    # every non-max key has P = 0.5312, just below the midpoint 0.53125 of the E4M3
    # neighbours 0.5 and 0.5625, so each rounds down by almost 2^-4 of itself; with
    # V > 0 all errors add up
    d, n = 1, 64
    scale = 1.0
    q = np.ones((1, d))
    k = np.full((n, d), math.log(0.5312))
    k[0] = 0.0
    v = np.linspace(1.0, 2.0, n)[:, None]
    vis = np.ones((1, n), bool)
    ob, _ = M.fp8_forward_bounds(q, k, v, scale, vis)
    o = M.exact_rows(q, k, v, scale, vis)[3]
    err = np.abs(M.simulate_fp8_forward(q, k, v, scale, vis) - o)
    assert np.all(err <= ob)
    assert err.max() / ob.max() > 0.8


def test_statistical_tolerance_catches_a_packing_mistake():
    # P values written to the wrong key inside each group of four (a plausible slip
    # when packing four 8-bit values per 32-bit column)
    inp = inputs.make_fp8_inputs(1, 1, 512, 128, seed=31)
    q, k, v, vis = _head(inp, 0, 0)
    o = M.exact_rows(q, k, v, inp.scale, vis)[3]
    perm = np.arange(512).reshape(-1, 4)[:, ::-1].reshape(-1)
    wrong = M.simulate_fp8_forward(q, k, v[perm], inp.scale, vis)
    assert M.rel_fro(wrong, o) > 10 * M.O_REL_FRO_TOL
