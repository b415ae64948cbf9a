"""Pins for the float64 oracle: each check compares it with something other
than itself -- the format definition, torch's float8 cast, an integer
rounding model, closed forms, the pages' alternative formulations of the same
attention (online softmax, split-KV combine, seesaw, ETAP transpose, weight
absorption) and brute force in plain Python floats.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import mla_oracle as om
import synth


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# e4m3 format
# ---------------------------------------------------------------------------
def test_e4m3_table_matches_torch_float8():
    """All 256 codes decode like torch.float8_e4m3fn (a library routine)."""
    ours = oracle.e4m3_value_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert nan_o.sum() == 2
    np.testing.assert_array_equal(ours[~nan_o], ref[~nan_r])
    assert ours[0x7E] == 448.0 and np.nanmax(ours) == oracle.E4M3_MAX


def test_e4m3_golden_codes(golden_dir):
    table = oracle.e4m3_value_table()
    n = 0
    for line in open(os.path.join(golden_dir, "e4m3_codes.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        code_s, val_s = line.split()[:2]
        code, val = int(code_s, 16), float(val_s)
        if math.isnan(val):
            assert math.isnan(table[code])
        else:
            assert table[code] == val and math.copysign(1, table[code]) == math.copysign(1, val)
            if abs(val) <= 448:
                assert oracle.e4m3_encode_rne(np.array([val], np.float32))[0] == code
        n += 1
    assert n >= 10


def _e4m3_rne_integer_model(y: np.ndarray) -> np.ndarray:
    """Round fp32 -> e4m3 by integer arithmetic on the fp32 fields (an
    independent model: no value table)."""
    bits = y.astype(np.float32).view(np.uint32).astype(np.int64)
    sign = (bits >> 31) & 1
    exp = (bits >> 23) & 0xFF
    man = bits & 0x7FFFFF
    m24 = np.where(exp == 0, man, man | (1 << 23))        # fp32 subnormals -> 0 below anyway
    e = np.where(exp == 0, -126, exp - 127)               # value = m24 * 2^(e-23)
    # quantum of the result: 2^(max(e,-6) - 3)  (e4m3 normals keep 3 mantissa bits,
    # subnormals share the 2^-9 quantum)
    qexp = np.maximum(e, -6) - 3
    shift = (qexp - (e - 23))                              # >= 20
    shift = np.minimum(shift, 62)
    n = m24 >> shift
    rem = m24 - (n << shift)
    half = np.int64(1) << (shift - 1)
    up = (rem > half) | ((rem == half) & ((n & 1) == 1))
    n = n + up
    # n * 2^qexp is the rounded magnitude; rebuild the code
    val = n.astype(np.float64) * np.exp2(qexp.astype(np.float64))
    val = np.minimum(val, 448.0)
    # encode exact e4m3 magnitude -> code
    code = np.zeros_like(n)
    nz = val > 0
    ev = np.floor(np.log2(np.where(nz, val, 1.0))).astype(np.int64)
    norm = nz & (ev >= -6)
    mant = np.where(norm, np.round((val / np.exp2(ev) - 1.0) * 8.0), 0).astype(np.int64)
    code = np.where(norm, ((ev + 7) << 3) | mant, code)
    sub = nz & (ev < -6)
    code = np.where(sub, np.round(val / 2.0 ** -9).astype(np.int64), code)
    return (code | (sign << 7)).astype(np.uint8)


@pytest.mark.parametrize("lo_exp,hi_exp", [(-16, -6), (-6, 3), (3, 10)])
def test_e4m3_encode_matches_integer_model(lo_exp, hi_exp):
    """Every fp32 whose exponent lies in [lo_exp, hi_exp) with mantissas on a
    fine stride (all ties and all rounding boundaries of e4m3 included)."""
    exps = np.arange(lo_exp + 127, hi_exp + 127, dtype=np.uint32)
    # the low 20 mantissa bits only matter through 'below/at/above half'; cover
    # every top-3-bit pattern with a dense set of low patterns
    low = np.unique(np.concatenate([np.arange(0, 1 << 20, 4099, dtype=np.uint32),
                                    np.array([0, 1, (1 << 19) - 1, 1 << 19, (1 << 19) + 1,
                                              (1 << 20) - 1], np.uint32)]))
    top = np.arange(8, dtype=np.uint32) << 20
    man = (top[:, None] | low[None, :]).ravel()
    for sgn in (0, 1):
        b = (np.uint32(sgn) << 31) | (exps[:, None] << 23) | man[None, :]
        y = b.ravel().view(np.float32)
        np.testing.assert_array_equal(oracle.e4m3_encode_rne(y), _e4m3_rne_integer_model(y))


def test_e4m3_encode_matches_torch_cast_in_range():
    y = np.random.default_rng(7).standard_normal(200000).astype(np.float32) * 100
    y = np.clip(y, -448, 448)
    ours = oracle.e4m3_encode_rne(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_saturates():
    y = np.array([448.0, 460.0, 1e6, -1e30, 3.0e38], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode_rne(y), [0x7E, 0x7E, 0x7E, 0xFE, 0x7E])


# ---------------------------------------------------------------------------
# 656-byte row
# ---------------------------------------------------------------------------
def _bf16_bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_golden_row(golden_dir):
    row = np.zeros(576, np.float32)
    row[0:4] = [448, -224, 1, 0.5]
    row[128:131] = [3.5, -3.5, 0.0625]
    row[384:387] = [1.0, 1.0625, 1.125]
    row[512] = 1.0
    row[575] = -2.0
    raw = oracle.quantize_kv_fp8(_bf16_bits(row)[None, :])[0]
    assert raw.shape == (656,)
    checks = 0
    for line in open(os.path.join(golden_dir, "quant_rows.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        off = int(parts[1])
        want = [int(x, 16) for x in parts[2:]]
        assert list(raw[off:off + len(want)]) == want, parts[0]
        checks += 1
    assert checks == 9
    # everything else of the latent is code 0
    mask = np.ones(512, bool)
    mask[[0, 1, 2, 3, 128, 129, 130, 384, 385, 386]] = False
    assert (raw[:512][mask] == 0).all()


def test_row_layout_sizes():
    """656 = 512 (e4m3) + 16 (4 fp32) + 128 (64 bf16) vs 576*2 = 1152 bf16;
    the saving is 43% ("FlashMLA 实战", §FP8 缓存怎么把 KV 压掉四成)."""
    assert oracle.FP8_ROW_BYTES == 512 + 4 * 4 + 64 * 2 == 656
    assert 576 * 2 == 1152
    assert round(100 * (1 - 656 / 1152)) == 43
    # 128K tokens x 62 layers: 8.7 GiB in bf16 -> about 5 GiB in fp8 (same section)
    assert round(128 * 1024 * 62 * 1152 / 2 ** 30, 1) == 8.7
    assert round(128 * 1024 * 62 * 656 / 2 ** 30) == 5


def test_quantize_roundtrip_error_bound_and_fields():
    rows = synth.make_latent_rows(64, seed=3, outlier_channels=4)
    bits = rows.view(torch.int16).numpy().view(np.uint16)
    raw = oracle.quantize_kv_fp8(rows)
    deq = oracle.dequantize_kv_fp8(raw)
    x = oracle.bf16_to_f64(bits)
    # RoPE bytes are the bf16 input verbatim
    assert (raw[:, 528:].view("<u2") == bits[:, 512:]).all()
    np.testing.assert_array_equal(deq[:, 512:], x[:, 512:])
    scale = raw[:, 512:528].copy().view("<f4").astype(np.float64)
    lat = x[:, :512].reshape(64, 4, 128)
    amax = np.abs(lat).max(axis=2)
    np.testing.assert_array_equal(scale, (amax.astype(np.float32) / np.float32(448)).astype(np.float64))
    # the block maximum maps to +-448 (code 0x7E / 0xFE)
    codes = raw[:, :512].reshape(64, 4, 128)
    arg = np.abs(lat).argmax(axis=2)
    top = np.take_along_axis(codes, arg[:, :, None], 2)[..., 0]
    assert np.isin(top, [0x7E, 0xFE]).all()
    # rounding error at most half an e4m3 quantum of y = x/scale
    y = (lat.astype(np.float32) / scale[:, :, None].astype(np.float32)).astype(np.float64)
    q = deq[:, :512].reshape(64, 4, 128) / scale[:, :, None]
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    assert (np.abs(q - y) <= 2.0 ** (e - 4) + 1e-12).all()


# ---------------------------------------------------------------------------
# V4.1 rows of 512 values: 528 bytes (e4m3 + UE8M0) and 288 bytes (e2m1 + e4m3)
# ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §八 '版本漂移', §十 format table)
# ---------------------------------------------------------------------------
def _golden_row(golden_dir, name):
    codes, deq = [], []
    for line in open(os.path.join(golden_dir, name)):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, off, *vals = line.split()
        if kind == "deq":
            deq.append((int(off), float(vals[0])))
        else:
            codes.append((int(off), [int(v, 16) for v in vals]))
    return codes, deq


def _check_golden(raw, deq_row, codes, deq, data_bytes):
    touched = np.zeros(data_bytes, bool)
    for off, want in codes:
        assert list(raw[off:off + len(want)]) == want, off
        if off < data_bytes:
            touched[off:off + len(want)] = True
    assert (raw[:data_bytes][~touched] == 0).all()
    for dim, v in deq:
        assert deq_row[dim] == v and math.copysign(1, deq_row[dim]) == math.copysign(1, v), dim


def test_fp8_528_golden_row(golden_dir):
    row = np.zeros(512, np.float32)
    row[0:4] = [1.0, -0.5, 0.3, 1.75]
    row[32:34] = [3.0, -2.0 ** -12]
    row[96] = 2.0 ** -16
    row[128:130] = [57344.0, 100.0]
    raw = oracle.quantize_kv_fp8_528(_bf16_bits(row)[None, :])[0]
    assert raw.shape == (528,)
    codes, deq = _golden_row(golden_dir, "fp8_528_row.txt")
    _check_golden(raw, oracle.dequantize_kv_fp8_528(raw[None])[0], codes, deq, 512)


def test_fp4_288_golden_row(golden_dir):
    row = np.zeros(512, np.float32)
    row[0:5] = [6.0, -1.0, 0.75, 2.5, 0.2]
    row[16:18] = [7.0, -0.3125]
    row[48:51] = [3072.0, 224.0, -1120.0]
    row[64] = 0.01
    raw = oracle.quantize_kv_fp4_288(_bf16_bits(row)[None, :])[0]
    assert raw.shape == (288,)
    codes, deq = _golden_row(golden_dir, "fp4_288_row.txt")
    _check_golden(raw, oracle.dequantize_kv_fp4_288(raw[None])[0], codes, deq, 256)


def test_v41_row_sizes():
    """528 = 512 e4m3 + 16 UE8M0 (one per 32 values); 288 = 512 e2m1 at two
    per byte + 32 e4m3 (one per 16 values) (拆解 §八, §十 table: 1/124 of the
    MHA cache per token)."""
    assert oracle.FP8_528_ROW_BYTES == 512 + 512 // 32 == 528
    assert oracle.FP4_288_ROW_BYTES == 512 // 2 + 512 // 16 == 288


def test_e2m1_table_is_the_format():
    """FP4 e2m1 magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 (the OCP
    microscaling definition), negated under the sign bit."""
    t = oracle.e2m1_value_table()
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(t[:8]) == mags
    assert list(-t[8:]) == mags
    assert math.copysign(1, t[8]) == -1
    for c, v in enumerate(t):
        assert oracle.e2m1_encode_rne(np.array([v]))[0] == c


def test_ue8m0_values():
    assert oracle.ue8m0_value(127) == 1.0
    assert oracle.ue8m0_value(0) == 2.0 ** -127
    assert oracle.ue8m0_value(254) == 2.0 ** 127
    assert np.isnan(oracle.ue8m0_value(255))


def _to_bf16_rows(x64):
    t = torch.tensor(x64, dtype=torch.float64).to(torch.bfloat16)
    assert (t.to(torch.float64).numpy() == x64).all()      # the test builds exact bf16 values
    return t


def test_fp8_528_grid_round_trip():
    """Rows built from chosen codes and scales, with one +-448 per block so
    that the chosen scale is the minimal one: quantising gives the bytes back."""
    rng = _rng(40)
    n = 24
    table = oracle.e4m3_value_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    codes = rng.choice(finite, size=(n, 16, 32))
    codes[:, :, 0] = rng.choice([0x7E, 0xFE], size=(n, 16))
    k = rng.integers(-20, 8, size=(n, 16))
    x = table[codes] * np.exp2(k.astype(np.float64))[:, :, None]
    raw = oracle.quantize_kv_fp8_528(_to_bf16_rows(x.reshape(n, 512)))
    np.testing.assert_array_equal(raw[:, :512], codes.reshape(n, 512).astype(np.uint8))
    np.testing.assert_array_equal(raw[:, 512:], (k + 127).astype(np.uint8))
    np.testing.assert_array_equal(oracle.dequantize_kv_fp8_528(raw), x.reshape(n, 512))


def test_fp4_288_grid_round_trip():
    """The same for the 288-byte rows: one +-6 per block makes the chosen
    e4m3 scale the minimal one."""
    rng = _rng(41)
    n = 24
    e2m1 = oracle.e2m1_value_table()
    e4m3 = oracle.e4m3_value_table()
    codes = rng.integers(0, 16, size=(n, 32, 16))
    codes[:, :, 3] = rng.choice([7, 15], size=(n, 32))
    sc = rng.integers(1, 0x7F, size=(n, 32))                # positive finite e4m3
    x = e2m1[codes] * e4m3[sc][:, :, None]
    raw = oracle.quantize_kv_fp4_288(_to_bf16_rows(x.reshape(n, 512)))
    flat = codes.reshape(n, 512).astype(np.uint8)
    np.testing.assert_array_equal(raw[:, :256], flat[:, 0::2] | (flat[:, 1::2] << 4))
    np.testing.assert_array_equal(raw[:, 256:], sc.astype(np.uint8))
    np.testing.assert_array_equal(oracle.dequantize_kv_fp4_288(raw), x.reshape(n, 512))


def _blocks_of_mixed_magnitude(rng, n, width):
    """bf16-exact rows whose blocks have magnitudes from 1e-30 to 1e30, with
    exact ties planted."""
    mag = 10.0 ** rng.uniform(-30, 30, size=(n, 512 // width, 1))
    x = rng.standard_normal((n, 512 // width, width)) * mag
    x[:, ::5, 1] = 0.0
    return torch.tensor(x.reshape(n, 512)).to(torch.bfloat16)


def test_fp8_528_brute_force():
    """Per block, brute force in plain Python floats: the scale is the least
    power of two that lets 448 cover amax, and each code is a nearest e4m3
    value to x / 2^k (ties: even mantissa)."""
    rng = _rng(42)
    rows = _blocks_of_mixed_magnitude(rng, 6, 32)
    raw = oracle.quantize_kv_fp8_528(rows)
    x = rows.to(torch.float64).numpy().reshape(6, 16, 32)
    table = [float(v) for v in oracle.e4m3_value_table()]
    for r in range(6):
        for j in range(16):
            blk = [float(v) for v in x[r, j]]
            amax = max(abs(v) for v in blk)
            k = -127
            while 448.0 * 2.0 ** k < amax:
                k += 1
            assert raw[r, 512 + j] == k + 127
            for i, v in enumerate(blk):
                y = v / 2.0 ** k
                c = int(raw[r, 32 * j + i])
                best = min(abs(t - y) for t in table if t == t)
                assert abs(table[c] - y) == best
                if best > 0:
                    ties = [cc for cc in range(256) if table[cc] == table[cc] and abs(table[cc] - y) == best
                            and (cc & 0x80) == (c & 0x80)]
                    if len(ties) > 1:
                        assert c % 2 == 0
                assert (c & 0x80 != 0) == (math.copysign(1, v) < 0)


def test_fp4_288_brute_force():
    rng = _rng(43)
    rows = _blocks_of_mixed_magnitude(rng, 6, 16)
    rows[:, 7] = 2.0 ** -140          # a bf16 subnormal in a block
    raw = oracle.quantize_kv_fp4_288(rows)
    x = rows.to(torch.float64).numpy().reshape(6, 32, 16)
    e4 = [float(v) for v in oracle.e4m3_value_table()[:0x7F]]
    e2 = [float(v) for v in oracle.e2m1_value_table()]
    for r in range(6):
        for j in range(32):
            blk = [float(v) for v in x[r, j]]
            amax = max(abs(v) for v in blk)
            ok = [c for c in range(0x7F) if 6.0 * e4[c] >= amax]
            want_sc = ok[0] if ok else 0x7E
            assert raw[r, 256 + j] == want_sc
            v_sc = e4[want_sc]
            for i, v in enumerate(blk):
                d = 16 * j + i
                c = int(raw[r, d // 2] >> (4 * (d % 2))) & 0xF
                y = v / v_sc if v_sc > 0 else 0.0
                dist = [abs(abs(e2[m]) - min(abs(y), 6.0)) for m in range(8)]
                best = min(dist)
                assert dist[c & 7] == best
                if dist.count(best) > 1:
                    assert (c & 7) % 2 == 0
                assert (c >> 3) == (1 if math.copysign(1, v) < 0 else 0)


def test_v41_quantise_error_bounds():
    """|x - deq| is at most half a quantum: 2^(e-4) for e4m3 (e the binade of
    x/2^k, at least -6) and half the e2m1 step times the scale for FP4,
    wherever no saturation happens."""
    rows = synth.make_latent_rows(32, seed=44, outlier_channels=4)[:, :512].contiguous()
    x = oracle.to_f64(rows)
    raw8 = oracle.quantize_kv_fp8_528(rows)
    d8 = oracle.dequantize_kv_fp8_528(raw8)
    k = raw8[:, 512:].astype(np.float64) - 127
    y = x.reshape(32, 16, 32) / np.exp2(k)[:, :, None]
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
    assert (np.abs(d8.reshape(32, 16, 32) - x.reshape(32, 16, 32)) <= np.exp2(e - 4 + k[:, :, None]) + 0).all()
    raw4 = oracle.quantize_kv_fp4_288(rows)
    d4 = oracle.dequantize_kv_fp4_288(raw4)
    v = oracle.e4m3_value_table()[raw4[:, 256:]]
    a = np.abs(x.reshape(32, 32, 16)) / v[:, :, None]
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))   # e2m1 spacing
    assert (np.abs(d4.reshape(32, 32, 16) - x.reshape(32, 32, 16)) <= step / 2 * v[:, :, None]).all()


# ---------------------------------------------------------------------------
# attention: closed forms and brute force
# ---------------------------------------------------------------------------
def test_single_key_closed_form():
    rng = _rng(1)
    q = rng.standard_normal((4, 576))
    k = rng.standard_normal((1, 576))
    out, lse = oracle.attend(q, k, 0.05)
    np.testing.assert_array_equal(out, np.repeat(k[:, :512], 4, 0))
    np.testing.assert_allclose(lse, 0.05 * (q @ k[0]), rtol=0, atol=1e-12)


def test_identical_keys_closed_form():
    rng = _rng(2)
    q = rng.standard_normal((3, 576))
    k = np.repeat(rng.standard_normal((1, 576)), 37, 0)
    out, lse = oracle.attend(q, k, 0.1)
    np.testing.assert_allclose(out, np.repeat(k[:1, :512], 3, 0), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, 0.1 * (q @ k[0]) + math.log(37), rtol=0, atol=1e-12)


def test_empty_visible_set_reading():
    out, lse = oracle.attend(np.ones((2, 576)), np.zeros((0, 576)), 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_brute_force_plain_python_tiny():
    """B=1, L<=4, hand-expanded with Python floats."""
    rng = _rng(3)
    d_k, d_v = 6, 4
    for L in range(1, 5):
        q = rng.standard_normal((2, d_k))
        k = rng.standard_normal((L, d_k))
        sc = 0.7
        out, lse = oracle.attend(q, k, sc, d_v=d_v)
        for h in range(2):
            s = [sc * sum(q[h, d] * k[t, d] for d in range(d_k)) for t in range(L)]
            w = [math.exp(x) for x in s]          # no max shift: tiny values
            z = sum(w)
            for d in range(d_v):
                ref = sum(w[t] * k[t, d] for t in range(L)) / z
                assert abs(out[h, d] - ref) < 1e-13
            assert abs(lse[h] - math.log(z)) < 1e-13


def test_softmax_weights_sum_to_one():
    rng = _rng(4)
    q = rng.standard_normal((8, 576))
    k = rng.standard_normal((300, 576)) * 3
    sc = 576 ** -0.5
    _, lse = oracle.attend(q, k, sc)
    w = np.exp(sc * (q @ k.T) - lse[:, None])
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# the pages' other formulations of the same attention
# ---------------------------------------------------------------------------
def _flash_decode(qv, K, scale, d_v):
    """Online softmax, one token at a time (拆解 page §五, flashDecode)."""
    m, l = -math.inf, 0.0
    acc = np.zeros(d_v)
    for j in range(K.shape[0]):
        s = scale * float(qv @ K[j])
        m_new = max(m, s)
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = math.exp(s - m_new)
        l = l * alpha + p
        acc = acc * alpha + p * K[j, :d_v]
        m = m_new
    return acc / l, m + math.log(l)


def test_online_softmax_matches_two_pass():
    rng = _rng(5)
    q = rng.standard_normal((3, 576))
    K = rng.standard_normal((130, 576)) * 2
    sc = 576 ** -0.5
    out, lse = oracle.attend(q, K, sc)
    for h in range(3):
        o, ls = _flash_decode(q[h], K, sc, 512)
        np.testing.assert_allclose(o, out[h], rtol=1e-12, atol=1e-13)
        assert abs(ls - lse[h]) < 1e-12


def test_split_kv_combine_matches_at_every_split_point():
    """m = max m_i; l = sum l_i e^{m_i - m}; o = sum o_i l_i e^{m_i - m} / l
    (拆解 page §七 'split-KV：把长序列切开')."""
    rng = _rng(6)
    q = rng.standard_normal((2, 576))
    K = rng.standard_normal((40, 576))
    sc = 0.05
    full_o, full_lse = oracle.attend(q, K, sc)
    for cut in range(1, 40):
        o1, lse1 = oracle.attend(q, K[:cut], sc)
        o2, lse2 = oracle.attend(q, K[cut:], sc)
        # (o_i, l_i, m_i) from (o_i, lse_i): l_i e^{m_i} = e^{lse_i}
        m = np.maximum(lse1, lse2)
        w1, w2 = np.exp(lse1 - m), np.exp(lse2 - m)
        o = (o1 * w1[:, None] + o2 * w2[:, None]) / (w1 + w2)[:, None]
        np.testing.assert_allclose(o, full_o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(m + np.log(w1 + w2), full_lse, rtol=0, atol=1e-12)


def test_seesaw_schedule_matches_two_pass():
    """Two KV blocks per round, O split into O_L / O_R with the cross-scaled
    updates of the 11-step seesaw schedule (拆解 page §七 'seesaw 调度')."""
    rng = _rng(7)
    q = rng.standard_normal(576)
    K = rng.standard_normal((64 * 6, 576)) * 1.5
    sc = 576 ** -0.5
    ref, _ = oracle.attend(q[None], K, sc)
    half = 256
    oL, oR = np.zeros(half), np.zeros(half)
    m, l = -math.inf, 0.0
    for r in range(0, K.shape[0], 128):
        K0, K1 = K[r:r + 64], K[r + 64:r + 128]
        p0 = sc * (K0 @ q)                            # step 1
        p1 = sc * (K1 @ q)                            # step 2
        m0 = max(m, p0.max())                         # step 3
        s0 = math.exp(m - m0) if m != -math.inf else 0.0
        p0 = np.exp(p0 - m0)                          # step 4
        oL = oL * s0 + p0 @ K0[:, :half]              # step 5
        m1 = max(m0, p1.max())                        # step 6
        s1 = math.exp(m0 - m1)
        p1 = np.exp(p1 - m1)                          # step 7
        oR = oR * (s0 * s1) + p1 @ K1[:, half:512]    # step 8
        p0 = p0 * s1                                  # step 9
        oR = oR + p0 @ K0[:, half:512]                # step 10
        oL = oL * s1 + p1 @ K1[:, :half]              # step 11
        l = l * s0 * s1 + p0.sum() + p1.sum()
        m = m1
    np.testing.assert_allclose(np.concatenate([oL, oR]) / l, ref[0], rtol=1e-12, atol=1e-13)


def test_etap_transposed_formulation_matches():
    """S^T = K Q^T, column softmax, O = (V^T P^T)^T, blockwise with
    O <- diag(e^{m - m_new}) O + V_j^T P_j^T, final (diag(1/l) O)^T read as
    dividing each query column by its l (FlashMLA-ETAP page, §2.2, §3.2)."""
    rng = _rng(8)
    Nq, N = 16, 300
    Q = rng.standard_normal((Nq, 576))
    K = rng.standard_normal((N, 576))
    sc = 576 ** -0.5
    ref, ref_lse = oracle.attend(Q, K, sc)
    O = np.zeros((512, Nq))
    l = np.zeros(Nq)
    m = np.full(Nq, -np.inf)
    for j in range(0, N, 64):
        Kj = K[j:j + 64]
        S_T = sc * (Kj @ Q.T)                        # [Bc, Nq]
        m_new = np.maximum(m, S_T.max(axis=0))
        P_T = np.exp(S_T - m_new[None, :])
        r = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        l = r * l + P_T.sum(axis=0)
        O = O * r[None, :] + Kj[:, :512].T @ P_T
        m = m_new
    out = (O / l[None, :]).T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m + np.log(l), ref_lse, rtol=0, atol=1e-12)


def test_weight_absorption_identity():
    """Naive per-head attention with k_i = [W^UK_i c; k^R], v_i = W^UV_i c equals
    absorbed q~_i = W^UK_i^T q^C_i (oracle.absorb_q) scored against [c; k^R],
    followed by o_i = W^UV_i . (attention-weighted c) (oracle.up_project)
    (拆解 page §六 '吸收'). d_h != d_c, so a transposed weight fails by shape."""
    rng = _rng(9)
    n_h, d_h, d_c, d_R, T = 4, 8, 16, 4, 11
    W_UK = rng.standard_normal((n_h, d_h, d_c))
    W_UV = rng.standard_normal((n_h, d_h, d_c))
    c = rng.standard_normal((T, d_c))
    kR = rng.standard_normal((T, d_R))
    qC = rng.standard_normal((n_h, d_h))
    qR = rng.standard_normal((n_h, d_R))
    sc = (d_h + d_R) ** -0.5
    cache = np.concatenate([c, kR], axis=1)                  # the latent row
    q_abs = np.concatenate([oracle.absorb_q(qC, W_UK), qR], axis=1)
    lat, lse = oracle.attend(q_abs, cache, sc, d_v=d_c)
    o_abs = oracle.up_project(lat, W_UV)
    for i in range(n_h):
        k_i = np.concatenate([c @ W_UK[i].T, kR], axis=1)   # [T, d_h + d_R]
        v_i = c @ W_UV[i].T                                  # [T, d_h]
        s = sc * (k_i @ np.concatenate([qC[i], qR[i]]))
        p = np.exp(s - s.max())
        o_naive = (p @ v_i) / p.sum()
        np.testing.assert_allclose(o_abs[i], o_naive, rtol=1e-12, atol=1e-12)
        assert abs(lse[i] - (s.max() + math.log(p.sum()))) < 1e-12


def test_absorption_batched_over_tokens():
    """absorb_q / up_project over a token axis equal the per-token, per-head
    matrix-vector products written out as loops."""
    rng = _rng(19)
    T, n_h, d_h, d_c = 3, 2, 5, 7
    W_UK = rng.standard_normal((n_h, d_h, d_c))
    W_UV = rng.standard_normal((n_h, d_h, d_c))
    qC = rng.standard_normal((T, n_h, d_h))
    ol = rng.standard_normal((T, n_h, d_c))
    qa, ou = oracle.absorb_q(qC, W_UK), oracle.up_project(ol, W_UV)
    for t in range(T):
        for i in range(n_h):
            for c in range(d_c):
                assert abs(qa[t, i, c] - sum(W_UK[i, d, c] * qC[t, i, d] for d in range(d_h))) < 1e-12
            for d in range(d_h):
                assert abs(ou[t, i, d] - sum(W_UV[i, d, c] * ol[t, i, c] for c in range(d_c))) < 1e-12


# ---------------------------------------------------------------------------
# paging, causality, sparsity
# ---------------------------------------------------------------------------
def _small_dense(seqlens, s_q=1, causal=False, seed=0, h_q=4):
    case = synth.make_dense_case(seqlens, s_q=s_q, h_q=h_q, causal=causal, seed=seed)
    q = oracle.to_f64(case.q)
    kv = oracle.to_f64(case.kv_rows)
    return case, q, kv


def test_block_table_gather_equals_contiguous():
    """A shuffled page order reached through the block table gives the same
    result as the same tokens stored contiguously."""
    case, q, kv = _small_dense([130, 64, 1], seed=11)
    out, lse, bad = oracle.mla_decode(q, kv, cache_seqlens=case.cache_seqlens.numpy(),
                                      block_table=case.block_table.numpy(), page_block=64)
    assert not bad
    bt = case.block_table.numpy()
    for b, L in enumerate(case.cache_seqlens.numpy()):
        rows = synth.paged_rows_index(bt[b], int(L), 64)
        o2, l2 = oracle.attend(q[b, 0], kv[rows], case.softmax_scale)
        np.testing.assert_array_equal(out[b, 0], o2)
        np.testing.assert_array_equal(lse[b, 0], l2)


def test_causal_bottom_right_reading():
    case, q, kv = _small_dense([70, 5], s_q=2, causal=True, seed=12)
    sl = case.cache_seqlens.numpy()
    out, lse, _ = oracle.mla_decode(q, kv, cache_seqlens=sl, block_table=case.block_table.numpy(),
                                    page_block=64, causal=True)
    bt = case.block_table.numpy()
    for b in range(2):
        for i in range(2):
            rows = synth.paged_rows_index(bt[b], int(sl[b]) - 1 + i, 64)
            o2, l2 = oracle.attend(q[b, i], kv[rows], case.softmax_scale)
            np.testing.assert_array_equal(out[b, i], o2)
    # non-causal: both query positions see every token
    out_nc, _, _ = oracle.mla_decode(q, kv, cache_seqlens=sl, block_table=bt, page_block=64)
    rows = synth.paged_rows_index(bt[0], int(sl[0]), 64)
    np.testing.assert_array_equal(out_nc[0, 0], oracle.attend(q[0, 0], kv[rows], case.softmax_scale)[0])


def test_sparse_equals_dense_over_selected_subset():
    rng = _rng(13)
    case, q, kv = _small_dense([200], seed=13)
    bt = case.block_table.numpy()
    rows_all = synth.paged_rows_index(bt[0], 200, 64)
    # indices = every token (no -1) -> the dense result
    idx = rows_all[None, None, :].astype(np.int32)
    o_s, l_s, _ = oracle.mla_decode(q, kv, indices=idx)
    o_d, l_d, _ = oracle.mla_decode(q, kv, cache_seqlens=case.cache_seqlens.numpy(), block_table=bt)
    np.testing.assert_array_equal(o_s, o_d)
    # a random subset padded with -1 -> dense attention over the compacted subset
    pick = rng.choice(200, size=50, replace=False)
    idx2 = np.full((1, 1, 64), -1, np.int32)
    slots = rng.choice(64, size=50, replace=False)
    idx2[0, 0, slots] = rows_all[pick]
    o2, l2, _ = oracle.mla_decode(q, kv, indices=idx2)
    compact = kv[rows_all[pick]]
    o3, l3 = oracle.attend(q[0, 0], compact, case.softmax_scale)
    np.testing.assert_allclose(o2[0, 0], o3, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l2[0, 0], l3, rtol=0, atol=1e-12)


def test_out_of_range_index_is_reported_and_skipped():
    case, q, kv = _small_dense([64], seed=14)
    idx = np.array([[[0, 5, kv.shape[0] + 3, -1, -7]]], np.int32)
    o, l, bad = oracle.mla_decode(q, kv, indices=idx)
    assert bad
    o2, l2 = oracle.attend(q[0, 0], kv[[0, 5]], case.softmax_scale)
    np.testing.assert_array_equal(o[0, 0], o2)
