"""Seeded input generator: determinism, bf16 rounding and mask recipes."""
import numpy as np
import torch

from io_aware_exact_attention_gb300 import inputs


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], np.float32)])
    x = x.astype(np.float32)
    ours = inputs.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(inputs.bf16_bits_to_f32(ours), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_inputs_are_deterministic_and_bf16_exact():
    a = inputs.workload_inputs("bert_large_padded", B=2, H=2, N=256)
    b = inputs.workload_inputs("bert_large_padded", B=2, H=2, N=256)
    for n in ("q", "k", "v", "dout"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
        np.testing.assert_array_equal(inputs.round_bf16(getattr(a, n)), getattr(a, n))
    assert not np.array_equal(a.q, a.k)
    assert a.kv_len.shape == (2,) and np.all((a.kv_len >= 256) & (a.kv_len <= 512))
    assert abs(float(a.q.std()) - 1.0) < 0.02


def test_block_mask_recipe():
    bm = inputs.make_block_mask(8192, band=4, global_cols=1, frac=0.10, seed=1005)
    t = 64
    assert bm.shape == (t, t) and bm.dtype == np.uint8
    i, j = np.indices((t, t))
    assert np.all(bm[np.abs(i - j) <= 4] == 1)
    assert np.all(bm[:, 0] == 1)
    base = int(((np.abs(i - j) <= 4) | (j == 0)).sum())
    assert base == 615
    assert base < int(bm.sum()) <= base + 410
    np.testing.assert_array_equal(bm, inputs.make_block_mask(8192, band=4, global_cols=1, frac=0.10, seed=1005))


def test_fp32_workload_not_rounded():
    a = inputs.workload_inputs("tiny_fp32")
    assert a.dtype == "fp32" and a.q.dtype == np.float32
    assert not np.array_equal(inputs.round_bf16(a.q), a.q)
    assert a.device_array("q") is a.q


def test_qk_inputs_shapes_determinism_and_rounding():
    a = inputs.make_qk_inputs(2, 3, 5, 300, 128, seed=4, kv_len_range=(10, 300))
    b = inputs.make_qk_inputs(2, 3, 5, 300, 128, seed=4, kv_len_range=(10, 300))
    assert a.q.shape == (2, 3, 5, 128) and a.k.shape == a.v.shape == (2, 3, 300, 128)
    for n in ("q", "k", "v"):
        x = getattr(a, n)
        np.testing.assert_array_equal(x, getattr(b, n))
        np.testing.assert_array_equal(inputs.round_bf16(x), x)  # bf16-exact
        np.testing.assert_array_equal(inputs.bf16_bits_to_f32(a.device_array(n)), x)
    assert a.kv_len.shape == (2,) and np.all((a.kv_len >= 10) & (a.kv_len <= 300))
    # Q uses the same stream as make_inputs with that seed
    sq = inputs.make_inputs(2, 3, 5, 128, seed=4, with_dout=False)
    np.testing.assert_array_equal(sq.q, a.q)
    for name, spec in inputs.QK_WORKLOADS.items():
        assert name in inputs.QK_WORKLOAD_SEEDS and spec["d"] == 128
