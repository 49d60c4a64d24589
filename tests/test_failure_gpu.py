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


# ---------------------------------------------------- production kernels' abort path

@pytest.fixture(scope="module")
def fault_lib():
    """The failure-path test build (5 ms wait limit; CTA 0 of the d = 128 bf16 and FP8
    forward and of the d = 128 backward skips one tile load), loaded beside the normal
    library.  Built here, on first use; the normal build does not contain it."""
    path = _lib.build(extra_flags=_lib.FAULT_TEST_FLAGS, lib_path=_lib.FAULT_TEST_LIB_PATH)
    return _lib.load_variant(path)


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _check_after_abort(inp, o_normal, lse_normal, what):
    ro, rl = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=inp.causal)
    parity.check_forward(parity.to_host64(o_normal), lse_normal.cpu().numpy().astype(np.float64), ro, rl, what=what)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_wait_timeout_drains_and_reports(fault_lib, causal):
    # 4 key tiles, so CTA 0's producer reaches the K tile it skips; its MMA issuers
    # wait for that tile, give up after 5 ms, drain their MMAs and the loads in
    # flight, release TMEM and exit; every other CTA completes normally
    inp = inputs.make_inputs(1, 2, 512, 128, seed=81, causal=causal, with_dout=False)
    q, k, v = (parity.to_device(inp, n) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 512), device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream().cuda_stream
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_OK
    rc = fault_lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), 1, 2, 512, 128, inp.scale, int(causal),
                          None, None, _lib.FA_BF16, stream)
    assert rc == _lib.FA_OK
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_ERR_TIMEOUT
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_OK  # reading cleared the word
    # the context is intact: the normal library's forward on the same inputs is exact
    o2, lse2 = fa.attention_forward(q, k, v, inp.scale, causal)
    assert fa.fa_get_device_status() == _lib.FA_OK
    _check_after_abort(inp, o2, lse2, "forward after an aborted call")


def test_backward_wait_timeout_drains_and_reports(fault_lib):
    # CTA 0 (key tile 0 of head 0) never gets its second dO tile: its MMA issuer gives
    # up, the drain warps finish their bulk reductions and stores, TMEM is released
    inp = inputs.make_inputs(1, 2, 512, 128, seed=82, causal=True)
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    o, lse = fa.attention_forward(q, k, v, inp.scale, True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = fa.new_workspace(q)
    stream = torch.cuda.current_stream().cuda_stream
    rc = fault_lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                          _ptr(ws), ws.numel(), 1, 2, 512, 128, inp.scale, 1, None, None, _lib.FA_BF16, stream)
    assert rc == _lib.FA_OK
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_ERR_TIMEOUT
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_OK
    # the normal library's backward afterwards matches the oracle
    dq2, dk2, dv2 = fa.attention_backward(q, k, v, o, lse, do, inp.scale, True)
    assert fa.fa_get_device_status() == _lib.FA_OK
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=True)
    h = parity.to_host64
    parity.check_grads({"dq": h(dq2), "dk": h(dk2), "dv": h(dv2)}, ref, what="backward after an aborted call")


def test_fp8_forward_wait_timeout_drains_and_reports(fault_lib):
    # the FP8 forward shares the producer hook: CTA 0's issuers give up on the K tile
    # that never arrives, drain and release TMEM; the normal FP8 forward afterwards is
    # held to the FP8 error model
    from tests import test_fp8_gpu as F
    inp = inputs.make_fp8_inputs(1, 2, 512, 128, seed=83, causal=True)
    dev, _, _ = F.to_dev(inp)
    o = torch.empty((1, 2, 512, 128), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((1, 2, 512), device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream().cuda_stream
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_OK
    ldv = int(dev["vt8"].stride(2))
    rc = fault_lib.fa_fwd_fp8(_ptr(dev["q8"]), _ptr(dev["k8"]), _ptr(dev["vt8"]), ldv, _ptr(o), _ptr(lse), 1, 2, 512,
                              128, inp.scale, inp.descale_q, inp.descale_k, inp.descale_v, 1, None, None, stream)
    assert rc == _lib.FA_OK
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_ERR_TIMEOUT
    assert fault_lib.fa_get_device_status(stream) == _lib.FA_OK
    o2, lse2 = F.run(inp)
    F.check_all(inp, o2, lse2)
