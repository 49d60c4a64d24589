"""Failure detection on the GPU without faulting or hanging it.

A self-test kernel waits on a barrier that nothing arrives on; its bounded wait
gives up after about a second, records FA_ERR_TIMEOUT in the device status word
and returns.  The host reads the status, the word is cleared, and the context
keeps working (a normal attention call afterwards is checked against the oracle).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import _lib, inputs
from tests import parity

pytestmark = pytest.mark.gpu


def test_stalled_wait_reports_timeout_and_context_survives():
    lib = _lib.load()
    assert fa.fa_get_device_status() == _lib.FA_OK
    t0 = time.perf_counter()
    assert lib.fa_selftest_wait_timeout(torch.cuda.current_stream().cuda_stream) == _lib.FA_OK
    status = fa.fa_get_device_status()
    elapsed = time.perf_counter() - t0
    assert status == _lib.FA_ERR_TIMEOUT
    assert 0.5 < elapsed < 30.0
    assert fa.fa_get_device_status() == _lib.FA_OK  # reading cleared the word

    inp = inputs.make_inputs(1, 2, 300, 64, seed=77, causal=True, with_dout=False)
    q, k, v = (parity.to_device(inp, n) for n in ("q", "k", "v"))
    o, lse = fa.attention_forward(q, k, v, inp.scale, True)
    assert fa.fa_get_device_status() == _lib.FA_OK
    ro, rl = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=True)
    parity.check_forward(parity.to_host64(o), lse.cpu().numpy().astype(np.float64), ro, rl, what="after timeout")


def test_host_side_errors_launch_nothing():
    inp = inputs.make_inputs(1, 1, 128, 64, seed=1, with_dout=False)
    q = parity.to_device(inp, "q")
    o = torch.full_like(q, float("nan"))
    lse = torch.empty((1, 1, 128), device="cuda", dtype=torch.float32)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q, q, q, o, lse, scale=-1.0)
    assert e.value.code == _lib.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all()  # nothing ran
