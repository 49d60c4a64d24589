"""Seeded synthetic inputs for the attention path and its oracle.

This module holds no attention arithmetic: it draws the operands, rounds them
to the storage type and builds the mask descriptions (key lengths, tile mask).
Both the CUDA path and the oracle consume exactly these arrays, so a parity test
compares arithmetic only.

Recipe (one numpy ``default_rng`` stream per tensor, spawned from one seed):
  * Q, K, V, dO ~ N(0, 1), drawn in float32, then rounded to bf16 with
    round-to-nearest-even (kept exact as float32 for the oracle, and as raw bf16
    bits for the device);
  * for the FP8 forward: the same float32 draws of Q, K, V, each divided by a
    power-of-two per-tensor scale (the smallest with max|x| / scale <= 448) and
    rounded to OCP FP8 E4M3 with round-to-nearest-even; the oracle gets
    code value * scale, which is exact;
  * key-padding lengths: integers uniform on [lo, hi], one per sequence;
  * block mask over 128x128 tiles: a local band of +-band tiles, the first tile
    column (global tokens) and a fraction of tiles drawn uniformly without
    replacement from all tiles.
The workloads below give the attention shapes of the pages' benchmarks (BERT-large
and GPT-2 training, long-range contexts, block-sparse attention); no dataset or
model weights are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

TILE = 128


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(x)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exactly equal float32 values."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value, returned as float32."""
    return bf16_bits_to_f32(bf16_bits(x))


E4M3_MAX = 448.0  # largest finite OCP FP8 E4M3 value (1.75 * 2^8); code 0x7F is NaN


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> OCP FP8 E4M3 codes (uint8: sign, 4 exponent bits with bias 7, 3
    mantissa bits), round to nearest even.  Magnitudes below 2^-6 use the subnormal
    step 2^-9.  Raises ValueError for NaN and for values that round past 448."""
    x = np.asarray(x, dtype=np.float32)
    if np.isnan(x).any():
        raise ValueError("NaN has no place in an E4M3 input")
    a = np.abs(x)
    _, e2 = np.frexp(a)                       # a = f * 2^e2 with f in [0.5, 1)
    e = np.maximum(e2 - 1, -6)                # binade exponent, clamped to the subnormal range
    # a * 2^(3 - e) is exact (a power-of-two scaling); rint rounds ties to even.  In
    # the subnormal range (e = -6) the same step 2^-9 applies and the code is the
    # multiple itself, which also carries into the first normal binade.
    q = np.rint(np.ldexp(a, 3 - e)).astype(np.int32)
    code = np.where(a < np.float32(2.0 ** -6), q, (e + 7) * 8 + (q - 8))
    if (code > 0x7E).any():
        raise ValueError("value beyond the E4M3 range (|x| rounds above 448)")
    return (code.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)).astype(np.uint8)


def _e4m3_values() -> np.ndarray:
    """Value of each of the 256 E4M3 codes: exponent field 0 gives m * 2^-9, otherwise
    (8 + m) * 2^(e - 10) = 1.m * 2^(e - 7); 0x7F and 0xFF are NaN."""
    c = np.arange(256, dtype=np.int32)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (8.0 + m) * np.exp2(e - 10.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag).astype(np.float32)


_E4M3_VALUES = _e4m3_values()


def e4m3_bits_to_f32(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 codes -> exactly equal float32 values (0x7F / 0xFF decode to NaN)."""
    return _E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def pow2_scale(x: np.ndarray) -> float:
    """Smallest power of two s with max|x| / s <= 448 (1.0 for an all-zero tensor)."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    if amax == 0.0:
        return 1.0
    return float(2.0 ** math.ceil(math.log2(amax / E4M3_MAX)))


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


@dataclass
class AttentionInputs:
    """Host copies of one workload's inputs.

    q, k, v, dout: float32 [B, H, N, d] holding bf16-exact values (or true fp32
    values when dtype == "fp32"); *_bits: the same values as bf16 bit patterns.
    """
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dout: np.ndarray
    dtype: str
    scale: float
    causal: bool
    kv_len: np.ndarray | None
    block_mask: np.ndarray | None
    seed: int
    bits: dict = field(default_factory=dict)

    def device_array(self, name: str) -> np.ndarray:
        """Array in the device storage type: uint16 bf16 bits, or float32."""
        a = getattr(self, name)
        if self.dtype == "fp32":
            return a
        if name not in self.bits:
            self.bits[name] = bf16_bits(a)
        return self.bits[name]


def make_block_mask(n: int, band: int, global_cols: int, frac: float, seed: int,
                    tile: int = TILE) -> np.ndarray:
    """uint8 [T, T] tile mask: |i - j| <= band, j < global_cols, plus round(frac*T*T)
    tiles drawn without replacement from all T*T tiles."""
    t = (n + tile - 1) // tile
    i = np.arange(t)[:, None]
    j = np.arange(t)[None, :]
    bm = (np.abs(i - j) <= band) | (j < global_cols)
    rng = _streams(seed, 7)[6]
    n_rand = int(round(frac * t * t))
    if n_rand:
        pick = rng.choice(t * t, size=n_rand, replace=False)
        bm.reshape(-1)[pick] = True
    return bm.astype(np.uint8)


def make_inputs(B: int, H: int, N: int, d: int, *, seed: int, dtype: str = "bf16",
                scale: float | None = None, causal: bool = False,
                kv_len_range: tuple[int, int] | None = None,
                block_mask: dict | None = None, with_dout: bool = True) -> AttentionInputs:
    """Draw Q, K, V, dO ~ N(0,1) and the mask description for one workload."""
    if dtype not in ("bf16", "fp32"):
        raise ValueError(dtype)
    rq, rk, rv, rdo, rlen, _rmask, _ = _streams(seed, 7)
    shape = (B, H, N, d)

    def draw(rng):
        x = rng.standard_normal(shape, dtype=np.float32)
        return x if dtype == "fp32" else round_bf16(x)

    q, k, v = draw(rq), draw(rk), draw(rv)
    dout = draw(rdo) if with_dout else np.zeros(shape, np.float32)
    kv_len = None
    if kv_len_range is not None:
        lo, hi = kv_len_range
        kv_len = rlen.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    bm = None
    if block_mask is not None:
        bm = make_block_mask(N, seed=seed, **block_mask)
    return AttentionInputs(q=q, k=k, v=v, dout=dout, dtype=dtype,
                           scale=(1.0 / math.sqrt(d)) if scale is None else float(scale),
                           causal=causal, kv_len=kv_len, block_mask=bm, seed=seed)


# The five workloads: shapes, masks and scale of the pages' benchmarks.
WORKLOADS = {
    "tiny_fp32": dict(B=1, H=1, N=128, d=64, dtype="fp32", scale=1 / 8, causal=False, fwd_only=True),
    "bert_large_padded": dict(B=16, H=16, N=512, d=64, dtype="bf16", scale=1 / 8, causal=False,
                              kv_len_range=(256, 512)),
    "gpt2_causal": dict(B=8, H=12, N=2048, d=64, dtype="bf16", scale=1 / 8, causal=True),
    "long_causal_16k": dict(B=1, H=32, N=16384, d=128, dtype="bf16", scale=1 / math.sqrt(128), causal=True),
    "long_causal_64k": dict(B=1, H=32, N=65536, d=128, dtype="bf16", scale=1 / math.sqrt(128), causal=True),
    "block_sparse_8k": dict(B=4, H=16, N=8192, d=64, dtype="bf16", scale=1 / 8, causal=False,
                            block_mask=dict(band=4, global_cols=1, frac=0.10)),
}

WORKLOAD_SEEDS = {
    "tiny_fp32": 1001, "bert_large_padded": 1002, "gpt2_causal": 1003,
    "long_causal_16k": 1004, "long_causal_64k": 1004, "block_sparse_8k": 1005,
}


@dataclass
class Fp8Inputs:
    """Host copies of one FP8 forward workload.

    q8, k8: E4M3 codes [B, H, N, d]; vt8: E4M3 codes of V transposed, [B, H, d, ldv]
    (key index fastest, row stride ldv >= N a multiple of 16, columns past N zero).
    q, k, v: float32 [B, H, N, d] holding code value * descale exactly -- the values
    the oracle receives."""
    q8: np.ndarray
    k8: np.ndarray
    vt8: np.ndarray
    ldv: int
    descale_q: float
    descale_k: float
    descale_v: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    scale: float
    causal: bool
    kv_len: np.ndarray | None
    block_mask: np.ndarray | None
    seed: int


def quantize_e4m3(x: np.ndarray) -> tuple[np.ndarray, float, np.ndarray]:
    """Per-tensor power-of-two scaling then E4M3 rounding: (codes, descale, x_q) with
    x_q = codes' values * descale (exact float32)."""
    s = pow2_scale(x)
    codes = e4m3_bits(np.asarray(x, np.float32) / np.float32(s))
    return codes, s, (e4m3_bits_to_f32(codes) * np.float32(s)).astype(np.float32)


def make_fp8_inputs(B: int, H: int, N: int, d: int, *, seed: int, scale: float | None = None,
                    causal: bool = False, kv_len_range: tuple[int, int] | None = None,
                    block_mask: dict | None = None) -> Fp8Inputs:
    """Q, K, V ~ N(0,1) (the float32 draws of make_inputs with the same seed), the same
    masks, quantized to E4M3 with one power-of-two scale per tensor."""
    raw = make_inputs(B, H, N, d, seed=seed, dtype="fp32", scale=scale, causal=causal,
                      kv_len_range=kv_len_range, block_mask=block_mask, with_dout=False)
    return fp8_inputs_from(raw)


def fp8_inputs_from(raw: AttentionInputs) -> Fp8Inputs:
    """FP8 inputs holding the float32 Q, K, V of `raw` (shape, masks and scale kept),
    each quantized to E4M3 with one power-of-two scale per tensor."""
    B, H, N, d = raw.q.shape
    q8, sq, q = quantize_e4m3(raw.q)
    k8, sk, k = quantize_e4m3(raw.k)
    v8, sv, v = quantize_e4m3(raw.v)
    ldv = max(16, (N + 15) // 16 * 16)
    vt8 = np.zeros((B, H, d, ldv), np.uint8)
    vt8[..., :N] = np.swapaxes(v8, 2, 3)
    return Fp8Inputs(q8=q8, k8=k8, vt8=vt8, ldv=ldv, descale_q=sq, descale_k=sk, descale_v=sv, q=q, k=k, v=v,
                     scale=raw.scale, causal=raw.causal, kv_len=raw.kv_len, block_mask=raw.block_mask,
                     seed=raw.seed)


def workload_fp8_inputs(name: str, *, seed: int | None = None, **override) -> Fp8Inputs:
    """FP8 inputs of a named workload (its shape, masks and scale; optionally with
    B/H/N overridden)."""
    spec = dict(WORKLOADS[name])
    for key in ("fwd_only", "dtype"):
        spec.pop(key, None)
    spec.update(override)
    return make_fp8_inputs(seed=WORKLOAD_SEEDS[name] if seed is None else seed, **spec)


@dataclass
class QKInputs:
    """Host copies of a query block against a separate key/value sequence (decode and
    chunked prefill): q float32 [B, H, Nq, d], k, v float32 [B, H, Nk, d], all holding
    bf16-exact values; no causal mask."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    scale: float
    kv_len: np.ndarray | None
    seed: int

    def device_array(self, name: str) -> np.ndarray:
        return bf16_bits(getattr(self, name))


def make_qk_inputs(B: int, H: int, Nq: int, Nk: int, d: int, *, seed: int, scale: float | None = None,
                   kv_len_range: tuple[int, int] | None = None) -> QKInputs:
    """Q ~ N(0,1) [B,H,Nq,d] and K, V ~ N(0,1) [B,H,Nk,d] rounded to bf16, one stream per
    tensor as in make_inputs; key lengths uniform on kv_len_range when given."""
    rq, rk, rv, _rdo, rlen, _rmask, _ = _streams(seed, 7)
    q = round_bf16(rq.standard_normal((B, H, Nq, d), dtype=np.float32))
    k = round_bf16(rk.standard_normal((B, H, Nk, d), dtype=np.float32))
    v = round_bf16(rv.standard_normal((B, H, Nk, d), dtype=np.float32))
    kv_len = None
    if kv_len_range is not None:
        lo, hi = kv_len_range
        kv_len = rlen.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    return QKInputs(q=q, k=k, v=v, scale=(1.0 / math.sqrt(d)) if scale is None else float(scale), kv_len=kv_len,
                    seed=seed)


# Split-KV workloads: a 128-row query block (chunked prefill, speculative decoding) and
# single-token decode against a 32k-token key/value cache, d = 128.
QK_WORKLOADS = {
    "prefill_chunk_32k": dict(B=4, H=32, Nq=128, Nk=32768, d=128),
    "decode_32k": dict(B=8, H=32, Nq=1, Nk=32768, d=128),
}
QK_WORKLOAD_SEEDS = {"prefill_chunk_32k": 1006, "decode_32k": 1007}


def qk_workload_inputs(name: str, **override) -> QKInputs:
    spec = dict(QK_WORKLOADS[name])
    spec.update(override)
    return make_qk_inputs(seed=QK_WORKLOAD_SEEDS[name], **spec)


def workload_inputs(name: str, *, seed: int | None = None, **override) -> AttentionInputs:
    """Inputs of a named workload (optionally with B/H/N overridden for small cases)."""
    spec = dict(WORKLOADS[name])
    spec.pop("fwd_only", None)
    spec.update(override)
    return make_inputs(seed=WORKLOAD_SEEDS[name] if seed is None else seed, **spec)
