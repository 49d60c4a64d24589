"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (a plugin whose host application owns all device memory, or a
latency-critical path that must not call cudaMalloc) get their scratch from a
fixed 64 MiB array inside the library instead of a caller-provided workspace.
These tests call the entry point through the C ABI and compare it with fa_bwd,
twice in a row, so the second call runs on scratch the first one left behind.
The file sorts last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import _lib, inputs
from tests import parity

pytestmark = pytest.mark.gpu

MAX_BYTES = 64 * 1024 * 1024


def noalloc_fn():
    lib = _lib.load()
    f = lib.fa_bwd_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, fl, i, vp, vp, i, vp]
    f.restype = i
    return f


def call_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale, causal, bm, kl):
    B, H, N, d = q.shape
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return noalloc_fn()(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv), B, H, N, d,
                        float(scale), int(causal), ptr(bm), ptr(kl), _lib.FA_BF16,
                        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,override", [("bert_large_padded", {}),
                                           ("gpt2_causal", dict(B=2, H=4, N=1000)),
                                           ("long_causal_16k", dict(H=2, N=3000))])
def test_matches_fa_bwd_on_two_calls_in_a_row(name, override):
    inp = inputs.workload_inputs(name, **override)
    q, k, v, do = (parity.to_device(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    o, lse = fa.attention_forward(q, k, v, inp.scale, inp.causal, bm, kl)
    ref = [t.float() for t in fa.attention_backward(q, k, v, o, lse, do, inp.scale, inp.causal, bm, kl)]
    B, H, N, d = q.shape
    assert fa.fa_bwd_workspace_size(B, H, N, d) <= MAX_BYTES
    for _ in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = call_noalloc(q, k, v, o, lse, do, dq, dk, dv, inp.scale, inp.causal, bm, kl)
        assert rc == _lib.FA_OK, _lib.status_string(rc)
        assert fa.fa_get_device_status() == 0
        for got, want, what in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            g, w = got.float().cpu().numpy(), want.cpu().numpy()
            assert np.all(np.isfinite(g)), what
            assert parity.rel_fro(g, w) <= parity.GRAD_REL_FRO, what
        # dK and dV involve no atomics: they must equal fa_bwd's bit for bit
        assert torch.equal(dk.float(), ref[1]) and torch.equal(dv.float(), ref[2])


def test_rejects_problems_beyond_the_scratch_size():
    # B*H*N = 262144 rows at d = 64 need 68 MB > 64 MiB; nothing is launched
    B, H, N, d = 1, 512, 512, 64
    assert fa.fa_bwd_workspace_size(B, H, N, d) > MAX_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, dtype=torch.float32, device="cuda")
    p = t.data_ptr()
    rc = noalloc_fn()(p, p, p, p, lse.data_ptr(), p, p, p, p, B, H, N, d, 0.125, 0, None, None, _lib.FA_BF16,
                      torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.FA_ERR_INVALID_ARG
