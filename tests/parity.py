"""Shared helpers for the GPU parity tests: device copies of the seeded inputs,
error metrics, and the tolerances of the method's numerical contract.

Tolerances (bf16 storage, fp32 accumulation), against the fp64 oracle:
  forward O:      max-abs <= 1e-2 and relative Frobenius <= 5e-3
  LSE (fp32):     max |dLSE| / max(|LSE|, 1) <= 1e-5
  gradients:      relative Frobenius <= 2e-2 for dQ, dK, dV
  fp32 forward:   relative Frobenius <= 1e-5, LSE as above
"""
from __future__ import annotations

import numpy as np
import torch

FWD_MAX_ABS = 1e-2
FWD_REL_FRO = 5e-3
LSE_REL = 1e-5
GRAD_REL_FRO = 2e-2
FP32_REL_FRO = 1e-5


def to_device(inp, name):
    a = inp.device_array(name)
    if inp.dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def masks_to_device(inp):
    bm = torch.from_numpy(inp.block_mask).cuda() if inp.block_mask is not None else None
    kl = torch.from_numpy(inp.kv_len).cuda() if inp.kv_len is not None else None
    return bm, kl


def to_host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(x, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def max_abs(x, ref):
    return float(np.max(np.abs(x - ref))) if x.size else 0.0


def lse_err(x, ref):
    """max |x - ref| / max(|ref|, 1) over rows with finite reference; -inf rows must match."""
    fin = np.isfinite(ref)
    if not np.array_equal(np.isneginf(x), np.isneginf(ref)):
        return float("inf")
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(x[fin] - ref[fin]) / np.maximum(np.abs(ref[fin]), 1.0)))


def check_forward(o, lse, ref_o, ref_lse, fp32=False, what=""):
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    e_fro = rel_fro(o, ref_o)
    e_lse = lse_err(lse, ref_lse)
    if fp32:
        assert e_fro <= FP32_REL_FRO, f"{what}: O rel-fro {e_fro:.3g}"
    else:
        e_abs = max_abs(o, ref_o)
        assert e_abs <= FWD_MAX_ABS, f"{what}: O max-abs {e_abs:.3g}"
        assert e_fro <= FWD_REL_FRO, f"{what}: O rel-fro {e_fro:.3g}"
    assert e_lse <= LSE_REL, f"{what}: LSE err {e_lse:.3g}"
    return e_fro, e_lse


def check_grads(got: dict, ref: dict, what=""):
    errs = {}
    for name in ("dq", "dk", "dv"):
        assert np.all(np.isfinite(got[name])), f"{what}: non-finite {name}"
        errs[name] = rel_fro(got[name], ref[name])
        assert errs[name] <= GRAD_REL_FRO, f"{what}: {name} rel-fro {errs[name]:.3g}"
    return errs
