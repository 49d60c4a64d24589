"""C ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every function include/fa_gb300.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

from io_aware_exact_attention_gb300 import _lib

HEADER = os.path.join(_lib.INCLUDE, "fa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    _lib.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_get_device_status", "fa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} not exported"


def test_status_strings_and_version(lib):
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(4) == b"FA_ERR_TIMEOUT"
    assert lib.fa_status_string(99) == b"FA_ERR_UNKNOWN"
    assert lib.fa_version() >= 100


def test_workspace_size_is_linear_in_n(lib):
    ws = [lib.fa_bwd_workspace_size(1, 32, n, 128) for n in (4096, 8192, 16384, 65536)]
    for n, w in zip((4096, 8192, 16384, 65536), ws):
        rows = 32 * n
        assert w == ((rows * 4 + 255) // 256) * 256 + ((rows * 128 * 4 + 255) // 256) * 256
    assert ws[3] == 16 * ws[0]
    # far below the N x N score matrix the method avoids (4096^2 fp32 = 67 MB per head)
    assert ws[0] < 4096 * 4096 * 4 * 32
    assert lib.fa_bwd_workspace_size(0, 1, 1, 64) == 0


A = 0x10000  # aligned fake device address: never dereferenced, every check below fails first


@pytest.mark.parametrize("args,expect", [
    (dict(d=32), _lib.FA_ERR_UNSUPPORTED),
    (dict(d=256), _lib.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), _lib.FA_ERR_UNSUPPORTED),
    (dict(B=-1), _lib.FA_ERR_INVALID_ARG),
    (dict(N=-5), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _lib.FA_ERR_INVALID_ARG),
    (dict(q=None), _lib.FA_ERR_INVALID_ARG),
    (dict(o=A + 8), _lib.FA_ERR_INVALID_ARG),
    (dict(lse=A + 2), _lib.FA_ERR_INVALID_ARG),
    (dict(B=1 << 20, H=1 << 12), _lib.FA_ERR_INVALID_ARG),
    (dict(N=0, q=None, k=None), _lib.FA_OK),
    (dict(B=0), _lib.FA_OK),
])
def test_fwd_rejects_bad_arguments_without_launching(lib, args, expect):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, scale=0.125, causal=0, block_mask=None,
              kv_len=None, dtype=_lib.FA_BF16, stream=None)
    kw.update(args)
    rc = lib.fa_fwd(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["B"], kw["H"], kw["N"], kw["d"], kw["scale"],
                    kw["causal"], kw["block_mask"], kw["kv_len"], kw["dtype"], kw["stream"])
    assert rc == expect


@pytest.mark.parametrize("args,expect", [
    (dict(d=64), _lib.FA_ERR_UNSUPPORTED),
    (dict(ldv=120), _lib.FA_ERR_INVALID_ARG),
    (dict(ldv=136), _lib.FA_ERR_INVALID_ARG),
    (dict(dq=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(dk=float("inf")), _lib.FA_ERR_INVALID_ARG),
    (dict(dv=-2.0), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=1e30, dq=1e30), _lib.FA_ERR_INVALID_ARG),  # the folded score scale overflows
    (dict(vt=A + 8), _lib.FA_ERR_INVALID_ARG),
    (dict(k=None), _lib.FA_ERR_INVALID_ARG),
    (dict(N=0, q=None), _lib.FA_OK),
])
def test_fwd_fp8_rejects_bad_arguments_without_launching(lib, args, expect):
    kw = dict(q=A, k=A, vt=A, ldv=128, B=1, H=1, N=128, d=128, scale=0.125, dq=1.0, dk=1.0, dv=1.0)
    kw.update(args)
    rc = lib.fa_fwd_fp8(kw["q"], kw["k"], kw["vt"], kw["ldv"], A, A, kw["B"], kw["H"], kw["N"], kw["d"], kw["scale"],
                        kw["dq"], kw["dk"], kw["dv"], 0, None, None, None)
    assert rc == expect


@pytest.mark.parametrize("args,expect", [
    (dict(d=64), _lib.FA_ERR_UNSUPPORTED),
    (dict(n_splits=0), _lib.FA_ERR_INVALID_ARG),
    (dict(n_splits=1025), _lib.FA_ERR_INVALID_ARG),
    (dict(Nk=-1), _lib.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=1000), _lib.FA_ERR_INVALID_ARG),
    (dict(ws=A + 4), _lib.FA_ERR_INVALID_ARG),
    (dict(k=None), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), _lib.FA_ERR_INVALID_ARG),
    (dict(Nq=0, q=None), _lib.FA_OK),
])
def test_fwd_splitkv_rejects_bad_arguments_without_launching(lib, args, expect):
    kw = dict(q=A, k=A, v=A, B=1, H=2, Nq=1, Nk=4096, d=128, scale=0.125, n_splits=4, ws=A)
    kw.update(args)
    ws_bytes = kw.get("ws_bytes", lib.fa_fwd_splitkv_workspace_size(1, 2, max(kw["Nq"], 1), 128, 4))
    rc = lib.fa_fwd_splitkv(kw["q"], kw["k"], kw["v"], A, A, kw["B"], kw["H"], kw["Nq"], kw["Nk"], kw["d"],
                            kw["scale"], None, kw["n_splits"], kw["ws"], ws_bytes, None)
    assert rc == expect


def test_splitkv_workspace_and_split_choice(lib):
    # two partials per chunk: float32 O rows and LSE, each 256-byte aligned
    for (B, H, Nq, n) in [(1, 1, 1, 1), (4, 32, 128, 2), (8, 32, 1, 4)]:
        rows = B * H * Nq * 2 * n
        assert lib.fa_fwd_splitkv_workspace_size(B, H, Nq, 128, n) == \
            ((rows * 128 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
    assert lib.fa_fwd_splitkv_workspace_size(1, 1, 1, 128, 0) == 0
    for (B, H, Nq, Nk) in [(8, 32, 1, 32768), (4, 32, 128, 32768), (1, 1, 128, 32768), (1, 1, 1, 300),
                           (64, 64, 2048, 256), (1, 1, 1, 1)]:
        n = lib.fa_fwd_splitkv_pick_splits(B, H, Nq, Nk)
        key_tiles = (Nk + 127) // 128
        assert 1 <= n <= max(1, (key_tiles + 1) // 2) and n <= 1024
    assert lib.fa_fwd_splitkv_pick_splits(0, 1, 1, 1) == 1


@pytest.mark.parametrize("args,expect", [
    (dict(dtype=_lib.FA_FP32), _lib.FA_ERR_UNSUPPORTED),
    (dict(d=96), _lib.FA_ERR_UNSUPPORTED),
    (dict(ws_bytes=100), _lib.FA_ERR_INVALID_ARG),
    (dict(ws=None), _lib.FA_ERR_INVALID_ARG),
    (dict(dq=A + 4), _lib.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), _lib.FA_ERR_INVALID_ARG),
    (dict(H=0), _lib.FA_OK),
])
def test_bwd_rejects_bad_arguments_without_launching(lib, args, expect):
    kw = dict(B=1, H=1, N=128, d=64, scale=0.125, dtype=_lib.FA_BF16, ws=A, dq=A)
    kw.update(args)
    ws_bytes = kw.get("ws_bytes", lib.fa_bwd_workspace_size(1, 1, 128, 64))
    rc = lib.fa_bwd(A, A, A, A, A, A, kw["dq"], A, A, kw["ws"], ws_bytes, kw["B"], kw["H"], kw["N"], kw["d"],
                    kw["scale"], 0, None, None, kw["dtype"], None)
    assert rc == expect


def test_stage_entry_points_validate(lib):
    assert lib.fa_bwd_preprocess(A, A, A, 10, 1, 1, 128, 64, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_postprocess(A + 1, A, 1 << 20, 1, 1, 128, 64, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_main(A, A, A, A, A, A, A, A, 1 << 20, 1, 1, 128, 48, 0.1, 0, None, None, None) == \
        _lib.FA_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU or eager fallback"):
        _lib.load()
