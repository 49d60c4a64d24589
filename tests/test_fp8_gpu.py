"""Parity of the FP8 forward (fa_fwd_fp8) with the fp64 oracle.

The oracle gets exactly the values the E4M3 codes and their scales stand for, so
the comparison measures the kernel's arithmetic.  That arithmetic rounds P to E4M3
for the P V product, so O is held to the error model in tests/fp8_error_model.py:
every element inside its bound, and a relative Frobenius error of at most 0.05
over the tensor; LSE is held to its own bound (score products only).  A case whose
probabilities are all exact in E4M3 (identical keys) is held to bf16 precision.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import fp8_error_model as M

pytestmark = pytest.mark.gpu


def to_dev(inp):
    dev = {n: torch.from_numpy(np.ascontiguousarray(getattr(inp, n))).cuda() for n in ("q8", "k8", "vt8")}
    bm = torch.from_numpy(inp.block_mask).cuda() if inp.block_mask is not None else None
    kl = torch.from_numpy(inp.kv_len).cuda() if inp.kv_len is not None else None
    return dev, bm, kl


def run(inp):
    dev, bm, kl = to_dev(inp)
    o, lse = fa.attention_forward_fp8(dev["q8"], dev["k8"], dev["vt8"], inp.scale, inp.descale_q, inp.descale_k,
                                      inp.descale_v, inp.causal, bm, kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check_head_rows(inp, o, lse, b, h, rows):
    """O and LSE of the given rows of head (b, h) against the oracle and the error bounds.
    Returns (sum of squared errors, sum of squared reference values) of O."""
    kl = None if inp.kv_len is None else int(inp.kv_len[b])
    N = inp.q.shape[2]
    ref = oracle.head_rows(inp.q[b, h], inp.k[b, h], inp.v[b, h], np.zeros_like(inp.q[b, h]), inp.scale,
                           causal=inp.causal, kv_len=kl, block_mask=inp.block_mask, rows=np.asarray(rows, np.int32))
    vis = M.visible(N, inp.causal, kl, inp.block_mask, rows)
    ob, lb = M.fp8_forward_bounds(inp.q[b, h][rows], inp.k[b, h], inp.v[b, h], inp.scale, vis)
    got_o, got_l = o[b, h][rows], lse[b, h][rows]
    err = np.abs(got_o - ref["o"])
    worst = np.unravel_index(np.argmax(err / ob), err.shape)
    assert np.all(err <= ob), f"head {b},{h} row {rows[worst[0]]} col {worst[1]}: |dO| {err[worst]:.3g} > {ob[worst]:.3g}"
    empty = ~vis.any(axis=1)
    assert np.all(np.isneginf(got_l[empty])) and np.all(got_o[empty] == 0)
    dl = np.abs(got_l[~empty] - ref["lse"][~empty])
    assert np.all(dl <= lb[~empty]), f"head {b},{h}: LSE error {dl.max():.3g}"
    return float(np.sum((got_o - ref["o"]) ** 2)), float(np.sum(ref["o"] ** 2))


def check_all(inp, o, lse):
    B, H, N, _ = inp.q.shape
    se = sr = 0.0
    for b in range(B):
        for h in range(H):
            e, r = check_head_rows(inp, o, lse, b, h, np.arange(N))
            se, sr = se + e, sr + r
    rel = (se / sr) ** 0.5
    assert rel <= M.O_REL_FRO_TOL, f"O rel-fro {rel:.3g}"
    return rel


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_ragged_tail(causal):
    inp = inputs.make_fp8_inputs(1, 2, 700, 128, seed=41, causal=causal)  # 5 full tiles + 60 rows
    o, lse = run(inp)
    rel = check_all(inp, o, lse)
    assert rel > 0.003  # P really is rounded to 8 bits (a bf16 P would give ~0.002)


def test_fp8_key_padding_with_empty_sequence():
    inp = inputs.make_fp8_inputs(3, 2, 520, 128, seed=42, kv_len_range=(130, 400))
    inp.kv_len = np.array([0, 333, 520], np.int32)  # no keys; mid-tile; all keys
    o, lse = run(inp)
    check_all(inp, o, lse)


def test_fp8_block_mask_with_empty_rows():
    inp = inputs.make_fp8_inputs(1, 2, 1024, 128, seed=43, block_mask=dict(band=1, global_cols=0, frac=0.1))
    inp.block_mask[2, :] = 0   # a query tile that sees nothing
    inp.block_mask[:, 5] = 0   # a key tile nobody sees
    o, lse = run(inp)
    check_all(inp, o, lse)


def test_fp8_causal_block_mask_and_padding():
    inp = inputs.make_fp8_inputs(2, 2, 900, 128, seed=46, causal=True, kv_len_range=(200, 900),
                                 block_mask=dict(band=1, global_cols=1, frac=0.3))
    inp.block_mask[3, :] = 0  # a query tile that sees nothing: its CTA partner still works
    o, lse = run(inp)
    check_all(inp, o, lse)


def test_fp8_identical_keys_exact_probabilities():
    # every visible key has the same score, so every P' is exactly 1 (exact in E4M3):
    # O_i = the mean of the visible V rows, to bf16 precision
    inp = inputs.make_fp8_inputs(1, 2, 384, 128, seed=44, causal=True)
    inp.k8[:] = inp.k8[:, :, :1, :]
    inp.k[:] = inp.k[:, :, :1, :]
    o, lse = run(inp)
    check_all(inp, o, lse)
    ref = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=True)
    n_vis = np.arange(1, 385, dtype=np.float64)
    mean_abs_v = np.cumsum(np.abs(inp.v.astype(np.float64)), axis=2) / n_vis[:, None]
    err = np.abs(o - ref[0])
    assert np.all(err <= 2.0 ** -8 * np.abs(ref[0]) + M.ACC_REL * mean_abs_v + 1e-6), f"max err {err.max():.3g}"
    assert np.allclose(ref[0], np.cumsum(inp.v.astype(np.float64), axis=2) / n_vis[:, None], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_running_max_jumps_between_key_tiles(causal):
    # Even query rows get a planted score component that jumps between key tiles
    # (natural log units 0, +5, +20, +28, -2 for key tiles 0..4).  The FP8 kernel's
    # offset then stays put within its 8-log2-unit slack (+5, for about 85% of the
    # rows; the rest move past it), moves with an O rescale (+20, +28) and falls
    # behind (-2).  Odd rows keep plain scores, so warps mix the cases.  The planted
    # values go through the same E4M3 quantization as the rest.
    N, d = 640, 128
    raw = inputs.make_inputs(1, 2, N, d, seed=951 + int(causal), dtype="fp32", causal=causal, with_dout=False)
    jump = np.array([0.0, 5.0, 20.0, 28.0, -2.0], np.float32)
    a = 8.0
    q, k = raw.q.copy(), raw.k.copy()
    q[:, :, 0::2, 0] = a
    q[:, :, 1::2, 0] = 0.0
    k[:, :, :, 0] = np.repeat(jump, 128)[None, None, :] * np.float32(np.sqrt(d) / a)
    inp = inputs.fp8_inputs_from(dataclasses.replace(raw, q=q, k=k))
    # the planted jumps survive quantization: mean planted score per key tile, even rows
    planted = inp.q[0, 0, 0::2, :1].astype(np.float64) @ inp.k[0, 0, :, :1].T.astype(np.float64) * inp.scale
    per_tile = planted.reshape(planted.shape[0], 5, 128).mean(axis=(0, 2))
    assert np.allclose(per_tile, jump, atol=0.5), per_tile
    o, lse = run(inp)
    check_all(inp, o, lse)


def test_fp8_rejects_bad_arguments():
    inp = inputs.make_fp8_inputs(1, 1, 128, 128, seed=45)
    dev, _, _ = to_dev(inp)
    o = torch.empty((1, 1, 128, 128), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((1, 1, 128), device="cuda", dtype=torch.float32)
    lib = fa._lib.load()
    ptr = [t.data_ptr() for t in (dev["q8"], dev["k8"], dev["vt8"])]
    stream = torch.cuda.current_stream().cuda_stream
    args = lambda ldv, d, ds: (ptr[0], ptr[1], ptr[2], ldv, o.data_ptr(), lse.data_ptr(), 1, 1, 128, d, 0.1, ds,
                               1.0, 1.0, 0, None, None, stream)
    assert lib.fa_fwd_fp8(*args(120, 128, 1.0)) == fa._lib.FA_ERR_INVALID_ARG   # ldv < N
    assert lib.fa_fwd_fp8(*args(136, 128, 1.0)) == fa._lib.FA_ERR_INVALID_ARG   # ldv not a multiple of 16
    assert lib.fa_fwd_fp8(*args(128, 64, 1.0)) == fa._lib.FA_ERR_UNSUPPORTED    # d = 64
    assert lib.fa_fwd_fp8(*args(128, 128, 0.0)) == fa._lib.FA_ERR_INVALID_ARG   # zero descale
    assert lib.fa_fwd_fp8(*args(128, 128, float("nan"))) == fa._lib.FA_ERR_INVALID_ARG


def test_fp8_long_causal_16k_sampled_rows():
    """The full 16k causal shape (B1 H32 N16384 d128) in one launch; sampled rows of
    sampled heads against the oracle, and the error model on them."""
    inp = inputs.workload_fp8_inputs("long_causal_16k")
    o, lse = run(inp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(16384 - 64, 16384),
                                     rng.choice(16384, 192, replace=False)]))
    se = sr = 0.0
    for h in (0, 13, 31):
        e, r = check_head_rows(inp, o, lse, 0, h, rows)
        se, sr = se + e, sr + r
    assert (se / sr) ** 0.5 <= M.O_REL_FRO_TOL
