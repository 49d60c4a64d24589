"""Out-of-bounds and missing-write checks for every entry point.

Each output and workspace buffer is placed in the middle of a larger allocation: a
4 KiB guard region on each side holds a canary byte pattern, and the interior is
filled with NaN bytes (0xFF) before the call.  After the call every guard byte
must be intact (nothing was written past either end) and every interior element
of the outputs must have been written (no NaN left; -inf LSE only for rows that
see no key).  The cases use ragged sizes, whose last tiles are partly past the
end of each tensor: the tile edge is 128 rows for queries and keys (the block
size of khetwal.com's worked example, section "A Worked Example in Pseudocode").
The results are also compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_attention_gb300 as fa
from io_aware_exact_attention_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

GUARD = 4096
_PATTERN = np.tile(np.array([0xA5, 0x5A, 0xC3, 0x3C], np.uint8), GUARD // 4)


class Guarded:
    """A tensor of `shape`/`dtype` inside [guard | interior | pad + guard] bytes."""

    def __init__(self, shape, dtype):
        elsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * elsize
        inner = (self.nbytes + 255) // 256 * 256
        self.buf = torch.empty(GUARD + inner + GUARD, dtype=torch.uint8, device="cuda")
        pat = torch.from_numpy(np.resize(_PATTERN, self.buf.numel())).cuda()
        self.buf.copy_(pat)
        self.buf[GUARD:GUARD + self.nbytes].fill_(0xFF)  # NaN in bf16 and fp32
        self.expect_tail = pat[GUARD + self.nbytes:].clone()
        self.expect_head = pat[:GUARD].clone()
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape) if self.nbytes else \
            torch.empty(shape, dtype=dtype, device="cuda")

    def guards_intact(self):
        return bool(torch.equal(self.buf[:GUARD], self.expect_head)) and \
            bool(torch.equal(self.buf[GUARD + self.nbytes:], self.expect_tail))


def _dev(inp, name):
    return parity.to_device(inp, name)


def _no_nan(t):
    return not bool(torch.isnan(t.float()).any())


CASES = [(N, d, causal) for N in (1, 127, 129, 200, 520) for d in (64, 128) for causal in (False, True)]


@pytest.mark.parametrize("N,d,causal", CASES)
def test_fwd_bwd_writes_stay_in_bounds(N, d, causal):
    inp = inputs.make_inputs(2, 2, N, d, seed=300 + N + d + int(causal), causal=causal,
                             kv_len_range=(1, N) if N > 1 else None)
    B, H = 2, 2
    q, k, v, do = (_dev(inp, n) for n in ("q", "k", "v", "dout"))
    bm, kl = parity.masks_to_device(inp)
    g = {n: Guarded((B, H, N, d), torch.bfloat16) for n in ("o", "dq", "dk", "dv")}
    g["lse"] = Guarded((B, H, N), torch.float32)
    g["ws"] = Guarded((fa.fa_bwd_workspace_size(B, H, N, d),), torch.uint8)
    fa.fa_fwd(q, k, v, g["o"].t, g["lse"].t, inp.scale, causal, bm, kl)
    fa.fa_bwd(q, k, v, g["o"].t, g["lse"].t, do, g["dq"].t, g["dk"].t, g["dv"].t, g["ws"].t, inp.scale, causal,
              bm, kl)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for name, gb in g.items():
        assert gb.guards_intact(), f"{name}: a guard byte was overwritten"
    for name in ("o", "dq", "dk", "dv", "lse"):
        assert _no_nan(g[name].t), f"{name}: an element was not written"
    # workspace: D for every row and the float32 dQ accumulator, all written
    rows = B * H * N
    ws = g["ws"].t
    dsum = ws[:rows * 4].view(torch.float32)
    acc_off = (rows * 4 + 255) // 256 * 256
    acc = ws[acc_off:acc_off + rows * d * 4].view(torch.float32)
    assert _no_nan(dsum) and _no_nan(acc)
    ref = oracle.attention_backward(inp.q, inp.k, inp.v, inp.dout, inp.scale, causal=causal, kv_len=inp.kv_len)
    h = parity.to_host64
    parity.check_forward(h(g["o"].t), g["lse"].t.cpu().numpy().astype(np.float64), ref["o"], ref["lse"],
                         what=f"N={N} d={d}")
    parity.check_grads({n: h(g[n].t) for n in ("dq", "dk", "dv")}, ref, what=f"N={N} d={d}")


@pytest.mark.parametrize("N", [1, 77, 200])
def test_fp32_forward_writes_stay_in_bounds(N):
    inp = inputs.make_inputs(1, 2, N, 64, seed=400 + N, dtype="fp32", with_dout=False)
    q, k, v = (_dev(inp, n) for n in ("q", "k", "v"))
    go, gl = Guarded((1, 2, N, 64), torch.float32), Guarded((1, 2, N), torch.float32)
    fa.fa_fwd(q, k, v, go.t, gl.t, inp.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    assert go.guards_intact() and gl.guards_intact()
    assert _no_nan(go.t) and _no_nan(gl.t)
    ro, rl = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale)
    parity.check_forward(parity.to_host64(go.t), gl.t.cpu().numpy().astype(np.float64), ro, rl, fp32=True)


@pytest.mark.parametrize("N,causal", [(129, False), (200, True)])
def test_fp8_forward_writes_stay_in_bounds(N, causal):
    inp = inputs.make_fp8_inputs(1, 2, N, 128, seed=500 + N, causal=causal)
    dev = {n: torch.from_numpy(np.ascontiguousarray(getattr(inp, n))).cuda() for n in ("q8", "k8", "vt8")}
    go, gl = Guarded((1, 2, N, 128), torch.bfloat16), Guarded((1, 2, N), torch.float32)
    fa.fa_fwd_fp8(dev["q8"], dev["k8"], dev["vt8"], go.t, gl.t, inp.scale, inp.descale_q, inp.descale_k,
                  inp.descale_v, causal)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    assert go.guards_intact() and gl.guards_intact()
    assert _no_nan(go.t) and _no_nan(gl.t)
    ro, _ = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=causal)
    # the FP8 path rounds P to E4M3; its tight element bounds are checked in
    # test_fp8_gpu.py, here only the coarse statistical tolerance of that file
    assert parity.rel_fro(parity.to_host64(go.t), ro) <= 0.05


@pytest.mark.parametrize("Nq,Nk,n_splits", [(1, 3000, 4), (77, 1000, 3), (200, 5000, 2)])
def test_splitkv_writes_stay_in_bounds(Nq, Nk, n_splits):
    inp = inputs.make_qk_inputs(2, 2, Nq, Nk, 128, seed=600 + Nq)

    def dev(n):
        return torch.from_numpy(inp.device_array(n).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev("q"), dev("k"), dev("v")
    go, gl = Guarded((2, 2, Nq, 128), torch.bfloat16), Guarded((2, 2, Nq), torch.float32)
    gw = Guarded((fa.fa_fwd_splitkv_workspace_size(2, 2, Nq, 128, n_splits),), torch.uint8)
    fa.fa_fwd_splitkv(q, k, v, go.t, gl.t, inp.scale, None, n_splits, gw.t)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    assert go.guards_intact() and gl.guards_intact() and gw.guards_intact()
    assert _no_nan(go.t) and _no_nan(gl.t)
    n = max(Nq, Nk)
    for b, h in ((0, 0), (1, 1)):
        qp = np.zeros((n, 128), np.float32)
        kp = np.zeros((n, 128), np.float32)
        vp = np.zeros((n, 128), np.float32)
        qp[:Nq], kp[:Nk], vp[:Nk] = inp.q[b, h], inp.k[b, h], inp.v[b, h]
        r = oracle.head_rows(qp, kp, vp, None, inp.scale, kv_len=Nk, rows=np.arange(Nq, dtype=np.int32))
        parity.check_forward(parity.to_host64(go.t[b, h]), gl.t[b, h].cpu().numpy().astype(np.float64),
                             r["o"], r["lse"], what=f"split-KV {Nq}x{Nk}")
