"""Python binding of the C ABI (include/fa_gb300.h).

Argument marshalling only: every step of the attention path runs in the CUDA
library.  Tensors are torch CUDA tensors (torch supplies device memory and the
current stream); the C entry points get raw pointers and sizes.  The functions
with C names take caller-allocated outputs; ``attention_forward`` /
``attention_backward`` allocate outputs and workspace with torch first.
"""
from __future__ import annotations

import torch

from . import _lib

_DTYPES = {torch.bfloat16: _lib.FA_BF16, torch.float32: _lib.FA_FP32}


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        detail = ""
        if self.code == _lib.FA_ERR_CUDA:
            detail = f" ({_lib.load().fa_last_cuda_error().decode()})"
        super().__init__(f"{where}: {_lib.status_string(code)}{detail}")


def _check(code: int, where: str):
    if code != _lib.FA_OK:
        raise FaError(code, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _same(ref, *ts):
    for t in ts:
        if t is not None and (t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous with equal shape and dtype")


def fa_fwd(q, k, v, o, lse, scale, causal=False, block_mask=None, kv_len=None, stream=None):
    """O, LSE <- attention(Q, K, V); all [B,H,N,d] contiguous CUDA tensors, lse [B,H,N] float32."""
    B, H, N, d = _shape(q)
    _same(q, k, v, o)
    if not q.is_contiguous() or lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("bad q or lse")
    dtype = _DTYPES.get(q.dtype)
    if dtype is None:
        raise ValueError(f"unsupported dtype {q.dtype}")
    code = _lib.load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                              int(bool(causal)), _ptr(block_mask), _ptr(kv_len), dtype, _stream(stream))
    _check(code, "fa_fwd")


_BYTE_TYPES = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t is not None)


def fa_fwd_fp8(q8, k8, vt8, o, lse, scale, descale_q, descale_k, descale_v, causal=False, block_mask=None,
               kv_len=None, stream=None):
    """O (bf16), LSE <- attention of E4M3 inputs with per-tensor scales.

    q8, k8: [B,H,N,d] uint8 or float8_e4m3fn; vt8: V transposed, [B,H,d,ldv] with a
    contiguous last dimension of stride 1 and rows ldv >= N (a multiple of 16) apart;
    o: bf16 [B,H,N,d]; lse: float32 [B,H,N]."""
    B, H, N, d = _shape(q8)
    if q8.dtype not in _BYTE_TYPES or k8.dtype != q8.dtype or vt8.dtype != q8.dtype:
        raise ValueError("q8, k8, vt8 must be uint8 or float8_e4m3fn tensors of one dtype")
    if tuple(k8.shape) != (B, H, N, d) or not q8.is_contiguous() or not k8.is_contiguous():
        raise ValueError("q8 and k8 must be contiguous [B, H, N, d]")
    if vt8.dim() != 4 or tuple(vt8.shape[:3]) != (B, H, d) or vt8.stride(3) != 1:
        raise ValueError("vt8 must be [B, H, d, ldv] with unit stride in the last dimension")
    ldv = int(vt8.stride(2))
    if vt8.shape[3] < N or vt8.stride(1) != d * ldv or vt8.stride(0) != H * d * ldv:
        raise ValueError("vt8 rows must hold at least N keys and be packed ldv apart")
    if o.dtype != torch.bfloat16 or tuple(o.shape) != (B, H, N, d) or not o.is_contiguous():
        raise ValueError("o must be contiguous bf16 [B, H, N, d]")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("bad lse")
    code = _lib.load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), ldv, _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                                  float(descale_q), float(descale_k), float(descale_v), int(bool(causal)),
                                  _ptr(block_mask), _ptr(kv_len), _stream(stream))
    _check(code, "fa_fwd_fp8")


def attention_forward_fp8(q8, k8, vt8, scale, descale_q, descale_k, descale_v, causal=False, block_mask=None,
                          kv_len=None, stream=None):
    """Allocate O (bf16) and LSE with torch and run fa_fwd_fp8.  Returns (o, lse)."""
    B, H, N, d = _shape(q8)
    o = torch.empty((B, H, N, d), device=q8.device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32)
    fa_fwd_fp8(q8, k8, vt8, o, lse, scale, descale_q, descale_k, descale_v, causal, block_mask, kv_len, stream)
    return o, lse


def fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits) -> int:
    return int(_lib.load().fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits))


def fa_fwd_splitkv_pick_splits(B, H, Nq, Nk) -> int:
    return int(_lib.load().fa_fwd_splitkv_pick_splits(B, H, Nq, Nk))


def fa_fwd_splitkv(q, k, v, o, lse, scale, kv_len=None, n_splits=None, workspace=None, stream=None):
    """O, LSE <- attention of Q [B,H,Nq,d] over K, V [B,H,Nk,d] (bf16, no causal mask),
    the keys of each query tile split into n_splits chunks whose partial results are
    merged by their log-sum-exp.  workspace: a uint8 CUDA tensor of at least
    fa_fwd_splitkv_workspace_size(...) bytes (allocated here when None)."""
    B, H, Nq, d = _shape(q)
    Nk = int(k.shape[2])
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("split-KV forward takes bf16 tensors")
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d]")
    _same(q, o)
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("bad lse")
    if n_splits is None:
        n_splits = fa_fwd_splitkv_pick_splits(B, H, Nq, Nk)
    if workspace is None:
        nbytes = fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits)
        workspace = torch.empty(max(nbytes, 16), device=q.device, dtype=torch.uint8)
    code = _lib.load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, float(scale),
                                      _ptr(kv_len), int(n_splits), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream))
    _check(code, "fa_fwd_splitkv")


def attention_forward_splitkv(q, k, v, scale, kv_len=None, n_splits=None, stream=None):
    """Allocate O and LSE (and the workspace) with torch and run fa_fwd_splitkv."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    fa_fwd_splitkv(q, k, v, o, lse, scale, kv_len, n_splits, None, stream)
    return o, lse


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(_lib.load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, scale, causal=False, block_mask=None, kv_len=None,
           stream=None):
    """dQ, dK, dV <- backward of attention for upstream gradient dO (bf16)."""
    B, H, N, d = _shape(q)
    _same(q, k, v, o, dout, dq, dk, dv)
    if q.dtype != torch.bfloat16:
        raise ValueError("backward takes bf16 tensors")
    code = _lib.load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, N, d,
                              float(scale), int(bool(causal)), _ptr(block_mask), _ptr(kv_len), _lib.FA_BF16,
                              _stream(stream))
    _check(code, "fa_bwd")


def fa_bwd_preprocess(o, dout, workspace, stream=None):
    B, H, N, d = _shape(o)
    code = _lib.load().fa_bwd_preprocess(_ptr(o), _ptr(dout), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), B, H, N, d, _stream(stream))
    _check(code, "fa_bwd_preprocess")


def fa_bwd_main(q, k, v, lse, dout, dk, dv, workspace, scale, causal=False, block_mask=None, kv_len=None,
                stream=None):
    B, H, N, d = _shape(q)
    code = _lib.load().fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dout), _ptr(dk), _ptr(dv),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, N, d,
                                   float(scale), int(bool(causal)), _ptr(block_mask), _ptr(kv_len), _stream(stream))
    _check(code, "fa_bwd_main")


def fa_bwd_postprocess(dq, workspace, stream=None):
    B, H, N, d = _shape(dq)
    code = _lib.load().fa_bwd_postprocess(_ptr(dq), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          B, H, N, d, _stream(stream))
    _check(code, "fa_bwd_postprocess")


def fa_get_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (0 = FA_OK)."""
    return int(_lib.load().fa_get_device_status(_stream(stream)))


def attention_forward(q, k, v, scale, causal=False, block_mask=None, kv_len=None, stream=None):
    """Allocate O and LSE with torch and run fa_fwd.  Returns (o, lse)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    fa_fwd(q, k, v, o, lse, scale, causal, block_mask, kv_len, stream)
    return o, lse


def new_workspace(q):
    B, H, N, d = _shape(q)
    nbytes = fa_bwd_workspace_size(B, H, N, d)
    return torch.empty(max(nbytes, 16), device=q.device, dtype=torch.uint8)


def attention_backward(q, k, v, o, lse, dout, scale, causal=False, block_mask=None, kv_len=None, workspace=None,
                       stream=None):
    """Allocate dQ, dK, dV (and the workspace if none is given) and run fa_bwd."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = new_workspace(q) if workspace is None else workspace
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, ws, scale, causal, block_mask, kv_len, stream)
    return dq, dk, dv
