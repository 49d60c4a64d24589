"""The C ABI calls captured in a CUDA graph and replayed.

A training or serving loop often captures its step once and replays it.  Every
argument of the attention calls (pointers, sizes, the tensor maps the host encodes)
is fixed at capture time, so replaying the graph after new values are written into
the captured input buffers must compute attention of the new values.  Both replays
are checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_forward_backward_replayed_from_a_cuda_graph(d, causal):
    B, H, N = 2, 2, 300
    cases = [inputs.make_inputs(B, H, N, d, seed=900 + s + d, causal=causal) for s in range(2)]
    q, k, v, do = (parity.to_device(cases[0], n) for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = fa.new_workspace(q)
    scale = cases[0].scale

    def step():
        fa.fa_fwd(q, k, v, o, lse, scale, causal)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, scale, causal)

    step()  # first calls on the device set kernel attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    h = parity.to_host64
    for inp in cases + cases[:1]:
        for name, t in (("q", q), ("k", k), ("v", v), ("dout", do)):
            t.copy_(parity.to_device(inp, name))
        o.fill_(float("nan"))
        dq.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == 0
        ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=causal)
        parity.check_forward(h(o), lse.cpu().numpy().astype(np.float64), ref["o"], ref["lse"], what="graph replay")
        parity.check_grads({"dq": h(dq), "dk": h(dk), "dv": h(dv)}, ref, what="graph replay")
