"""Plain float64 CPU oracle for MLA decode over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg. It shares no code with the CUDA library and
never calls it.

What it computes, and where the pages say so
----------------------------------------------
* Attention is the plain definition softmax(q k^T * scale) V, computed in two
  passes with the full score row materialised ("矩阵、注意力与 GPU：拆解 DeepGEMM
  与 FlashMLA", §五 '注意力：两个 GEMM 加一个 softmax'; FlashAttention is an IO
  reordering of exactly this, not an approximation, same section).
* After weight absorption every head scores the same 576-wide cache row,
  score = q~ . c + q^R . k^R, and the value is the 512-wide latent c itself
  (same page, §六 '结果：decode 变成 MQA'); so keys are whole rows and values
  are their first 512 entries.
* Paged addressing: token t of request b lives in page block_table[b][t//64],
  slot t%64 ("FlashMLA 实战", §最小调用: block_table, cache_seqlens).
* Sparse mode: indices[b, i, :] are absolute rows (page*page_block + offset),
  -1 marks an unused slot (拆解 page, §八 '当前 master 已经是稀疏注意力').
* FP8 row: 512 e4m3 values quantised per 128 with one fp32 scale each, then 4
  fp32 scales, then the 64 RoPE dims kept as bf16; 656 bytes ("FlashMLA 实战",
  §FP8 缓存怎么把 KV 压掉四成; 拆解 page §八 '格式').
* V4.1 rows (拆解 page §八 '版本漂移', §十 format table): 528 bytes = 512 e4m3
  values then 16 UE8M0 scales (2^(byte-127), one per 32 values, RoPE part
  quantised too); the FP4 option, 288 bytes = 512 e2m1 values two to a byte
  then 32 e4m3 scales (one per 16 values). These rows hold 512 values in all,
  so a V4.1 key is 512 wide and its value is the whole row (d_k = d_v = 512).

Readings where the pages are silent:
* causal with s_q > 1 is bottom-right aligned: query i of s_q sees tokens
  t <= L - s_q + i;
* an empty visible set gives out = 0 and lse = -inf;
* lse is natural-log, includes softmax_scale;
* the quantiser works in fp32: scale = amax / 448 (IEEE division, 1.0 if the
  block is all zero), code = e4m3 round-to-nearest-even of x / scale,
  saturated to +-448;
* an out-of-range index or page entry is skipped (and reported).
* the 528-byte quantiser: the scale is the smallest power of two 2^k
  (k >= -127) with 448 * 2^k >= amax (the pages' UE8M0 rule: a power-of-two
  scale rounded up, 拆解 page §三), code = e4m3 round-to-nearest-even of x/2^k;
* the 288-byte quantiser: the scale is the smallest non-negative e4m3 value v
  with 6 v >= amax (rounded up, like the UE8M0 scale), 448 when none is large
  enough (values then saturate to +-6); code = e2m1 round-to-nearest-even of
  x/v with the sign of x; value 2i in the low nibble of byte i.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
something other than itself (closed forms, the pages' other formulations,
brute force, torch's float8 cast, an integer rounding model).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence, Tuple

import numpy as np

E4M3_MAX = 448.0
FP8_ROW_BYTES = 656
_LAT = 512
_ROPE = 64
_DK = _LAT + _ROPE


# ----------------------------------------------------------------------------
# dtype helpers (bit-level; no rounding happens here)
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_f64(t) -> np.ndarray:
    """A torch tensor (bf16/fp16/fp32/...) or array -> float64 numpy (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                return bf16_to_f64(t.view(torch.int16).numpy().view(np.uint16))
            return t.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


# ----------------------------------------------------------------------------
# E4M3 (FP8, 'fn' variant: bias 7, no infinities, S.1111.111 = NaN, max 448)
# ----------------------------------------------------------------------------
def e4m3_value_table() -> np.ndarray:
    """Value of each of the 256 e4m3 codes, from the format's definition."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = math.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_POS_VALUES = e4m3_value_table()[:0x7F]   # codes 0x00..0x7E: 0 .. 448, increasing


def e4m3_encode_rne(y: np.ndarray) -> np.ndarray:
    """fp32 values -> e4m3 codes: nearest representable value, ties to the code
    with an even last mantissa bit, magnitudes above 448 saturated to 448.

    Works on magnitudes by locating the two neighbouring representable
    values in the sorted table of non-negative codes; the sign bit is then
    copied from the input (so -0.0 and small negatives give 0x80).
    """
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64))
    sat = a >= E4M3_MAX
    hi = np.searchsorted(_POS_VALUES, a, side="left")        # first value >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _POS_VALUES[hi], hi, code)           # exact hits
    code = np.where(sat, 0x7E, code).astype(np.uint8)
    neg = np.signbit(y)
    return np.where(neg, code | 0x80, code).astype(np.uint8)


# ----------------------------------------------------------------------------
# 656-byte FP8 cache rows
# ----------------------------------------------------------------------------
def quantize_kv_fp8(rows) -> np.ndarray:
    """bf16 cache rows [N, 576] -> uint8 [N, 656].

    Per 128-value block of the 512 latent dims: amax = max |x| (exact in fp32),
    scale = fp32(amax / 448) (1.0 for an all-zero block), code =
    e4m3_rne(fp32(x / scale)). Bytes [512, 528) are the 4 scales as
    little-endian fp32, bytes [528, 656) the 64 RoPE dims copied bit-for-bit
    as bf16 ("FlashMLA 实战", §FP8 缓存怎么把 KV 压掉四成).
    """
    import torch
    if isinstance(rows, torch.Tensor):
        assert rows.dtype == torch.bfloat16
        bits = rows.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    else:
        bits = np.asarray(rows, dtype=np.uint16)
    n = bits.shape[0]
    assert bits.shape[1] == _DK
    lat = (bits[:, :_LAT].astype(np.uint32) << 16).view(np.float32).reshape(n, 4, 128)
    amax = np.max(np.abs(lat), axis=2)
    scale = np.where(amax == 0, np.float32(1.0), amax / np.float32(E4M3_MAX)).astype(np.float32)
    y = (lat / scale[:, :, None]).astype(np.float32)
    codes = e4m3_encode_rne(y).reshape(n, _LAT)
    out = np.empty((n, FP8_ROW_BYTES), dtype=np.uint8)
    out[:, :_LAT] = codes
    out[:, _LAT:_LAT + 16] = scale.astype("<f4").view(np.uint8).reshape(n, 16)
    out[:, _LAT + 16:] = np.ascontiguousarray(bits[:, _LAT:]).astype("<u2").view(np.uint8).reshape(n, 128)
    return out


def dequantize_kv_fp8(raw: np.ndarray) -> np.ndarray:
    """uint8 [N, 656] -> float64 [N, 576]: e4m3 value x its block's fp32 scale
    (exact in float64), RoPE bf16 -> float64 (exact)."""
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    n = raw.shape[0]
    table = e4m3_value_table()
    vals = table[raw[:, :_LAT]].reshape(n, 4, 128)
    scale = raw[:, _LAT:_LAT + 16].copy().view("<f4").astype(np.float64).reshape(n, 4)
    out = np.empty((n, _DK), dtype=np.float64)
    out[:, :_LAT] = (vals * scale[:, :, None]).reshape(n, _LAT)
    out[:, _LAT:] = bf16_to_f64(raw[:, _LAT + 16:].copy().view("<u2"))
    return out


# ----------------------------------------------------------------------------
# V4.1 cache rows of 512 values: 528 bytes (e4m3 + UE8M0) and 288 bytes (e2m1 + e4m3)
# ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §八 '版本漂移' and the §十 format
# table: 512 fp8 values and 16 UE8M0 scales with the RoPE part quantised too;
# the FP4 option, 512 e2m1 values two to a byte and 32 e4m3 scales; data first,
# scales after; §三 'UE8M0': a power-of-two scale, rounded up)
# ----------------------------------------------------------------------------
V41_DIM = 512
FP8_528_ROW_BYTES = 528
FP4_288_ROW_BYTES = 288
E2M1_MAX = 6.0


def e2m1_value_table() -> np.ndarray:
    """Value of each of the 16 e2m1 (FP4) codes, from the format's definition:
    sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no inf or NaN."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        vals[code] = sign * ((m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))
    return vals


def ue8m0_value(byte) -> np.ndarray:
    """UE8M0 scale byte -> 2^(byte - 127); 0xFF is NaN."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.exp2((b - 127).astype(np.float64)))


def _rows_bf16_f64(rows, width: int) -> np.ndarray:
    """bf16 rows (torch tensor or uint16 bit patterns) [N, width] -> float64."""
    import torch
    if isinstance(rows, torch.Tensor):
        assert rows.dtype == torch.bfloat16
        bits = rows.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    else:
        bits = np.asarray(rows, dtype=np.uint16)
    assert bits.shape[-1] == width
    return bf16_to_f64(bits.reshape(-1, width))


def quantize_kv_fp8_528(rows) -> np.ndarray:
    """bf16 rows [N, 512] -> uint8 [N, 528].

    Per 32-value block j: amax = max |x|; the scale is the smallest power of
    two 2^k, k >= -127, with 448 * 2^k >= amax (so no value saturates); byte
    512 + j holds k + 127. Byte d holds e4m3_rne(x_d / 2^k), the division
    being exact.
    """
    x = _rows_bf16_f64(rows, V41_DIM)
    n = x.shape[0]
    blocks = x.reshape(n, 16, 32)
    amax = np.max(np.abs(blocks), axis=2)
    ks = np.arange(-127, 128)
    fits = E4M3_MAX * np.exp2(ks.astype(np.float64))[None, None, :] >= amax[:, :, None]
    k = ks[np.argmax(fits, axis=2)]                    # first k that fits
    y = blocks / np.exp2(k.astype(np.float64))[:, :, None]
    out = np.empty((n, FP8_528_ROW_BYTES), dtype=np.uint8)
    out[:, :V41_DIM] = e4m3_encode_rne(y.astype(np.float32)).reshape(n, V41_DIM)
    out[:, V41_DIM:] = (k + 127).astype(np.uint8)
    return out


def dequantize_kv_fp8_528(raw: np.ndarray) -> np.ndarray:
    """uint8 [N, 528] -> float64 [N, 512]: e4m3 value x 2^(byte - 127) of its
    32-value block (exact in float64)."""
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    n = raw.shape[0]
    vals = e4m3_value_table()[raw[:, :V41_DIM]].reshape(n, 16, 32)
    scale = ue8m0_value(raw[:, V41_DIM:])
    return (vals * scale[:, :, None]).reshape(n, V41_DIM)


_E2M1_POS = e2m1_value_table()[:8]                     # 0, .5, 1, 1.5, 2, 3, 4, 6


def e2m1_encode_rne(y: np.ndarray) -> np.ndarray:
    """float64 values -> e2m1 codes: nearest magnitude, ties to the code with an
    even last bit, magnitudes above 6 saturated to 6; the sign bit copied from
    the input."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    d_lo = a - _E2M1_POS[lo]
    d_hi = _E2M1_POS[hi] - a
    code = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)), hi, lo)
    code = np.where(a >= E2M1_MAX, 7, code)
    return np.where(np.signbit(y), code | 0x8, code).astype(np.uint8)


def quantize_kv_fp4_288(rows) -> np.ndarray:
    """bf16 rows [N, 512] -> uint8 [N, 288].

    Per 16-value block j: the scale is the smallest non-negative e4m3 value v
    with 6 v >= amax (the block's largest value then needs no saturation), or
    448 when no e4m3 value is large enough; byte 256 + j holds its code. Each
    value becomes e2m1_rne(x / v) (0 with the sign of x when v = 0); byte i
    holds value 2i in its low nibble and value 2i + 1 in its high nibble.
    """
    x = _rows_bf16_f64(rows, V41_DIM)
    n = x.shape[0]
    blocks = x.reshape(n, 32, 16)
    amax = np.max(np.abs(blocks), axis=2)
    fits = E2M1_MAX * _POS_VALUES[None, None, :] >= amax[:, :, None]   # codes 0x00..0x7E
    sc = np.where(fits.any(axis=2), np.argmax(fits, axis=2), 0x7E).astype(np.uint8)
    v = _POS_VALUES[sc]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(v[:, :, None] > 0, blocks / np.where(v > 0, v, 1.0)[:, :, None], 0.0 * blocks)
    codes = e2m1_encode_rne(y).reshape(n, V41_DIM)
    out = np.empty((n, FP4_288_ROW_BYTES), dtype=np.uint8)
    out[:, :256] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    out[:, 256:] = sc
    return out


def dequantize_kv_fp4_288(raw: np.ndarray) -> np.ndarray:
    """uint8 [N, 288] -> float64 [N, 512]: e2m1 value x the e4m3 scale of its
    16-value block (exact in float64)."""
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    n = raw.shape[0]
    codes = np.empty((n, V41_DIM), dtype=np.uint8)
    codes[:, 0::2] = raw[:, :256] & 0xF
    codes[:, 1::2] = raw[:, :256] >> 4
    vals = e2m1_value_table()[codes].reshape(n, 32, 16)
    scale = e4m3_value_table()[raw[:, 256:]]
    return (vals * scale[:, :, None]).reshape(n, V41_DIM)


# ----------------------------------------------------------------------------
# the per-head GEMMs around attention (weight absorption)
# ----------------------------------------------------------------------------
def absorb_q(q_nope, w_uk) -> np.ndarray:
    """Absorbed query q~_{t,i} = W^UK_i^T q^C_{t,i} ("矩阵、注意力与 GPU：拆解
    DeepGEMM 与 FlashMLA", §六 '吸收'), so that q~ . c equals q^C . (W^UK c).
    q_nope [..., h, d_h], w_uk [h, d_h, d_c] -> [..., h, d_c], float64."""
    return np.einsum("hdc,...hd->...hc", np.asarray(w_uk, np.float64), np.asarray(q_nope, np.float64))


def up_project(o_lat, w_uv) -> np.ndarray:
    """Per-head output o_{t,i} = W^UV_i o~_{t,i} from the attention-weighted
    latent o~ (same section: the value is W^UV_i c, and the weights sum
    commutes with W^UV_i). o_lat [..., h, d_c], w_uv [h, d_h, d_c] ->
    [..., h, d_h], float64."""
    return np.einsum("hdc,...hc->...hd", np.asarray(w_uv, np.float64), np.asarray(o_lat, np.float64))


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def attend(qh: np.ndarray, keys: np.ndarray, scale: float, d_v: int = _LAT
           ) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention of one query position against a set of key rows.

    qh   [h, d_k] float64 (one row per head)
    keys [T, d_k] float64 (shared by all heads; the value is keys[:, :d_v])
    returns out [h, d_v], lse [h] (natural log, includes ``scale``).

    Two passes with the whole score row materialised: S = q K^T * scale,
    m = max S, P = exp(S - m), l = sum P, out = P V / l, lse = m + ln l.
    """
    qh = np.asarray(qh, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    h = qh.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((h, d_v)), np.full(h, -np.inf)
    s = (qh @ keys.T) * scale
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    l = p.sum(axis=1)
    out = (p @ keys[:, :d_v]) / l[:, None]
    return out, m + np.log(l)


def visible_rows(b: int, i: int, *, seqlens=None, block_table=None, page_block: int = 64,
                 s_q: int = 1, causal: bool = False, indices=None,
                 num_rows: Optional[int] = None) -> Tuple[np.ndarray, bool]:
    """Absolute cache rows that query i of request b attends to, and whether
    an out-of-range page/index had to be dropped.

    Dense: tokens 0 .. L_vis-1 with L_vis = L (non-causal) or L - s_q + 1 + i
    (causal, bottom-right aligned), through the block table. Sparse: the
    entries of indices[b, i] that are not -1, in their given order.
    """
    bad = False
    if indices is not None:
        sel = np.asarray(indices[b, i], dtype=np.int64)
        sel = sel[sel != -1]
        if num_rows is not None:
            ok = (sel >= 0) & (sel < num_rows)
            bad = bool((~ok).any())
            sel = sel[ok]
        return sel, bad
    L = int(seqlens[b])
    if causal:
        L = L - s_q + 1 + i
    L = max(L, 0)
    t = np.arange(L, dtype=np.int64)
    pages = np.asarray(block_table[b], dtype=np.int64)[t // page_block] if L else np.zeros(0, np.int64)
    rows = pages * page_block + t % page_block
    if num_rows is not None and L:
        ok = (pages >= 0) & (rows < num_rows)
        bad = bool((~ok).any())
        rows = rows[ok]
    return rows, bad


def mla_decode(q, kv_rows, *, cache_seqlens=None, block_table=None, page_block: int = 64,
               softmax_scale: Optional[float] = None, causal: bool = False, indices=None,
               d_v: int = _LAT, heads: Optional[Sequence[int]] = None):
    """Reference decode over every (request, query position).

    q        [B, s_q, h_q, d_k] float64
    kv_rows  [num_rows, d_k] float64 -- the cache viewed as rows
             (page p, slot j is row p*page_block + j)
    returns out [B, s_q, h, d_v], lse [B, s_q, h], any_bad_index
    """
    q = np.asarray(q, dtype=np.float64)
    B, s_q, h_q, d_k = q.shape
    if softmax_scale is None:
        softmax_scale = d_k ** -0.5
    hsel = list(range(h_q)) if heads is None else list(heads)
    out = np.zeros((B, s_q, len(hsel), d_v))
    lse = np.zeros((B, s_q, len(hsel)))
    any_bad = False
    n = kv_rows.shape[0]
    for b in range(B):
        for i in range(s_q):
            rows, bad = visible_rows(b, i, seqlens=cache_seqlens, block_table=block_table,
                                     page_block=page_block, s_q=s_q, causal=causal,
                                     indices=indices, num_rows=n)
            any_bad |= bad
            o, ls = attend(q[b, i, hsel], kv_rows[rows], softmax_scale, d_v)
            out[b, i], lse[b, i] = o, ls
    return out, lse, any_bad
