"""The standard-attention comparison leg of the benchmark (S and P materialised in
HBM, cuBLAS GEMMs and PyTorch softmax) against the fp64 oracle.

It is a baseline, not part of the library, and it keeps S and P in bf16 as a
framework does for bf16 inputs, so its tolerance is looser than the tiled path's:
rounding S (|S| of a few units) and P to bf16 moves each probability by up to
2^-8 of itself, and a relative Frobenius error of O up to 2e-2 (gradients 5e-2)
leaves room for that.  The test only has to show that the comparison computes
the same attention, so that its timings are timings of the same result."""
import numpy as np
import pytest
import torch

import bench
import oracle
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,d,causal", [(256, 64, False), (300, 128, True), (1024, 128, True)])
def test_standard_attention_matches_oracle(N, d, causal):
    inp = inputs.make_inputs(1, 2, N, d, seed=700 + N + d, causal=causal)
    q, k, v, do = (parity.to_device(inp, n).requires_grad_(n != "dout") for n in ("q", "k", "v", "dout"))
    o = bench.standard_attention(torch, q, k, v, inp.scale, causal)
    o.backward(do)
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=causal)
    h = parity.to_host64
    assert parity.rel_fro(h(o), ref["o"]) <= 2e-2
    for name, t in (("dq", q), ("dk", k), ("dv", v)):
        assert parity.rel_fro(h(t.grad), ref[name]) <= 5e-2, name


def test_sweep_row_reports_memory_and_time():
    import io_aware_exact_attention_gb300 as fa
    flush = bench.L2Flush(torch)
    row = bench.time_standard_vs_tiled(torch, fa, flush, 2048, H=4, steps=2, warmup=1)
    for key in ("standard_fwd_ms", "tiled_fwd_ms", "standard_fwd_bwd_ms", "tiled_fwd_bwd_ms"):
        assert row[key] > 0
    # the standard path holds at least the N x N scores of every head; the tiled path
    # holds O(N d) per head (O, LSE, and for the backward dQ, dK, dV and the workspace)
    assert row["standard_fwd_peak_bytes"] >= 4 * 2048 * 2048 * 2
    assert row["tiled_fwd_bwd_peak_bytes"] < row["standard_fwd_peak_bytes"]
