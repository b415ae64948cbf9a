"""GPU parity for the V4.1 cache rows of 512 values ("矩阵、注意力与 GPU：拆解
DeepGEMM 与 FlashMLA", §八 '版本漂移' and the §十 format table): 528-byte rows
(512 e4m3 + 16 UE8M0 scales, one per 32) and 288-byte FP4 rows (512 e2m1 two
to a byte + 32 e4m3 scales, one per 16). A V4.1 key is the whole 512-value
row, and so is its value.

* The quantisers are compared with the oracle's byte for byte, on random rows,
  on blocks of extreme and tiny magnitude, on exact ties and on every finite
  bf16 bit pattern.
* Decode (paged and token-sparse, split and unsplit, causal s_q = 2) is
  compared with the oracle run on the oracle's dequantised rows.
* Gathering is exact: with one key per query dominating by about 196 log2
  units (the others' weights underflow fp32), the output is that key's
  dequantised row bit for bit.
* A UE8M0 scale beyond 2^7, a query entry beyond fp16's range and halves of
  a score more than about 22 binades apart are reported as MLA_ERR_RANGE.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import assert_close_attn

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")

DEV = "cuda"
MLA_ERR_RANGE = 7
FORMATS = {
    "fp8_528": dict(fmt=2, row=528, quant=lambda x: mla.mla_quantize_kv_fp8_528(x),
                    oq=oracle.quantize_kv_fp8_528, odq=oracle.dequantize_kv_fp8_528),
    "fp4_288": dict(fmt=3, row=288, quant=lambda x: mla.mla_quantize_kv_fp4_288(x),
                    oq=oracle.quantize_kv_fp4_288, odq=oracle.dequantize_kv_fp4_288),
}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


# ---------------------------------------------------------------------------
# quantisers
# ---------------------------------------------------------------------------
def _special_rows():
    """Rows with blocks of every kind: zeros, +-0, bf16 subnormals, tiny and
    huge magnitudes, values on the e4m3 / e2m1 grids and exactly between them."""
    rows = []
    rng = np.random.default_rng(90)
    for mag in [0.0, 2.0 ** -133, 1e-30, 1e-6, 1e-2, 1.0, 7.0, 448.0, 2688.0, 3000.0, 1e6, 3e7, 1e30]:
        rows.append(rng.standard_normal(512) * mag)
    z = np.zeros(512)
    z[::3] = -0.0
    rows.append(z)
    grid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1.0])  # e2m1 midpoints and values
    rows.append(np.resize(np.concatenate([grid, -grid]), 512) * 2.0 ** rng.integers(-3, 4, size=512))
    e4 = oracle.e4m3_value_table()
    e4 = e4[np.isfinite(e4)]
    mids = (np.sort(e4)[1:] + np.sort(e4)[:-1]) / 2                        # e4m3 ties
    rows.append(np.resize(mids, 512))
    return torch.tensor(np.stack(rows)).to(torch.bfloat16)


def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32)
    e = (bits >> 7) & 0xFF
    bits = bits[e != 0xFF].astype(np.uint16)                                  # no inf / NaN
    bits = np.resize(bits, (len(bits) + 511) // 512 * 512)
    return torch.from_numpy(bits.view(np.int16).reshape(-1, 512)).view(torch.bfloat16)


@pytest.mark.parametrize("name", list(FORMATS))
@pytest.mark.parametrize("kind", ["random", "special", "all_bf16"])
def test_quantiser_bit_exact(name, kind):
    f = FORMATS[name]
    if kind == "random":
        rows = synth.make_latent_rows(1000, seed=91, outlier_channels=4, d_k=512)
    elif kind == "special":
        rows = _special_rows()
    else:
        rows = _all_finite_bf16()
    got = f["quant"](rows.to(DEV)).cpu().numpy()
    want = f["oq"](rows)
    assert got.shape == want.shape == (rows.shape[0], f["row"])
    if not np.array_equal(got, want):
        r, c = np.argwhere(got != want)[0]
        raise AssertionError(f"{name}/{kind}: {int((got != want).sum())} bytes differ; first row {r} byte {c}: "
                             f"gpu {got[r, c]:#04x} oracle {want[r, c]:#04x}")


def test_quantiser_empty():
    assert mla.mla_quantize_kv_fp8_528(torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)).shape == (0, 528)
    assert mla.mla_quantize_kv_fp4_288(torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)).shape == (0, 288)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
def _meta(sl, s_q, fmt, *, causal=False, batch=None, topk=0, parts=None):
    if topk:
        return mla.mla_get_metadata(None, s_q, 128, batch=batch, topk=topk, kv_format=fmt, device=DEV,
                                    num_sm_parts=parts)
    return mla.mla_get_metadata(sl, s_q, 128, causal=causal, kv_format=fmt, num_sm_parts=parts)


def _run_dense(case, f, parts=None):
    raw = f["quant"](case.kv_rows.to(DEV))
    sl = case.cache_seqlens.to(DEV)
    meta, ns = _meta(sl, case.s_q, f["fmt"], causal=case.causal, parts=parts)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(DEV), raw.view(case.num_blocks, 64, 1, f["row"]),
                                           case.block_table.to(DEV), sl, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, causal=case.causal, kv_format=f["fmt"])
    torch.cuda.synchronize()
    return raw, out, lse, mla.mla_read_status(device=DEV)


def _oracle_dense(case, raw, f):
    deq = f["odq"](raw.cpu().numpy())
    out, lse, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, cache_seqlens=case.cache_seqlens.numpy(),
                                    block_table=case.block_table.numpy(), softmax_scale=case.softmax_scale,
                                    causal=case.causal)
    return out, lse


@pytest.mark.parametrize("name", list(FORMATS))
@pytest.mark.parametrize("lens,s_q,causal,parts", [
    ((200, 77, 1, 130), 1, False, None),       # ragged tails, a 1-token request
    ((200, 77, 1, 130), 1, False, 3),          # every request cut into pieces (split + combine)
    ((333, 64, 129), 2, True, None),           # two query positions, bottom-right causal
    ((0, 150), 1, False, None),                # an empty request: out 0, lse -inf
])
def test_dense_parity(name, lens, s_q, causal, parts):
    f = FORMATS[name]
    case = synth.make_dense_case(list(lens), s_q=s_q, causal=causal, seed=92, outlier_channels=4, d_k=512)
    raw, out, lse, (st, bits) = _run_dense(case, f, parts)
    assert st == 0, (st, bits)
    ro, rl = _oracle_dense(case, raw, f)
    assert_close_attn(out, lse, ro, rl, f"{name} dense {lens} s_q={s_q} causal={causal} parts={parts}")


@pytest.mark.parametrize("name", list(FORMATS))
@pytest.mark.parametrize("s_q,topk", [(1, 192), (2, 160)])
def test_sparse_parity(name, s_q, topk):
    f = FORMATS[name]
    case = synth.make_sparse_case(3, s_q, topk, tokens_per_request=1024, seed=93, outlier_channels=4, d_k=512)
    raw = f["quant"](case.kv_rows.to(DEV))
    meta, ns = _meta(None, s_q, f["fmt"], batch=3, topk=topk)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(DEV), raw.view(-1, 64, 1, f["row"]), None, None, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, kv_format=f["fmt"],
                                           indices=case.indices.to(DEV))
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, (st, bits)
    deq = f["odq"](raw.cpu().numpy())
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, indices=case.indices.numpy(),
                                  softmax_scale=case.softmax_scale)
    assert_close_attn(out, lse, ro, rl, f"{name} sparse s_q={s_q} topk={topk}")


def _exact_rows(n, seed, fp4):
    """bf16 rows on the format's grid whose every block holds its full-scale
    value, so that quantising reproduces them and every dequantised value is
    exact in bf16: 528 -- blocks of 32 with amax 7 = 448 * 2^-6; 288 -- blocks
    of 16 with amax 6 (scale 1)."""
    g = np.random.default_rng(seed)
    if fp4:
        mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
        x = g.choice(mags, size=(n, 512)) * g.choice([-1.0, 1.0], size=(n, 512))
        x.reshape(n, 32, 16)[:, :, 5] = 6.0
    else:
        x = np.clip(g.standard_normal((n, 512)), -6.5, 6.5)
        x.reshape(n, 16, 32)[:, :, 9] = -7.0
    return torch.tensor(x).to(torch.bfloat16)


def _signal_dims(c):
    """Four dims in each half of the pair (c < 64)."""
    return [c + 64 * j for j in range(4)] + [256 + c + 64 * j for j in range(4)]


def _plant_dominant(rows, q, row, qi, c):
    """Row `row` dominates query position qi (all heads) through the 8 dims of
    _signal_dims(c): 8 * 64 * 6 / sqrt(512) * log2(e), about 196 log2 units,
    with every other row at most 0 there once their positive values in these
    dims are cleared; the others' weights 2^-196 are below fp32's range."""
    for d in _signal_dims(c):
        rows[row, d] = 6.0
        q[qi][..., d] = 64.0


def _clear_others(rows, dom, c_of):
    """Zero the positive values of every row in each query's signal dims,
    except in that query's dominant row."""
    for key, r in dom.items():
        keep = rows[r].clone()
        for d in _signal_dims(c_of(key)):
            col = rows[:, d]
            col[col > 0] = 0
        rows[r] = keep


@pytest.mark.parametrize("name", list(FORMATS))
def test_sparse_gather_exact(name):
    f = FORMATS[name]
    fp4 = name == "fp4_288"
    B, s_q, topk, nrows = 3, 2, 96, 4096
    rows = _exact_rows(nrows, 94, fp4)
    rng = np.random.default_rng(95)
    idx = np.stack([np.stack([rng.choice(nrows, size=topk, replace=False) for _ in range(s_q)]) for _ in range(B)])
    idx = idx.astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    q = torch.zeros(B, s_q, 128, 512, dtype=torch.bfloat16)
    dom = {}
    for b in range(B):
        for i in range(s_q):
            valid = np.flatnonzero(idx[b, i] >= 0)
            r = int(idx[b, i, rng.choice(valid)])
            _plant_dominant(rows, q, r, (b, i), (b * s_q + i) % 64)
            dom[(b, i)] = r
    assert len(set(dom.values())) == len(dom)
    _clear_others(rows, dom, lambda key: (key[0] * s_q + key[1]) % 64)
    raw = f["quant"](rows.to(DEV))
    deq = f["odq"](raw.cpu().numpy())
    want = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(want.double().numpy(), deq)
    meta, ns = _meta(None, s_q, f["fmt"], batch=B, topk=topk)
    mla.mla_read_status(device=DEV)
    out, _ = mla.mla_decode_with_kvcache(q.to(DEV), raw.view(-1, 64, 1, f["row"]), None, None, 512, meta, ns,
                                         kv_format=f["fmt"], indices=torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, (st, bits)
    for (b, i), r in dom.items():
        assert torch.equal(out[b, i].cpu(), want[r].unsqueeze(0).expand(128, 512)), (b, i)


@pytest.mark.parametrize("name", list(FORMATS))
def test_paged_gather_exact(name):
    f = FORMATS[name]
    fp4 = name == "fp4_288"
    case = synth.make_dense_case([200, 130, 64], seed=96, d_k=512)
    rows = _exact_rows(case.kv_rows.shape[0], 97, fp4)
    q = torch.zeros_like(case.q)
    bt = case.block_table.numpy()
    dom = {}
    for b, L in enumerate([200, 130, 64]):
        toks = synth.paged_rows_index(bt[b], L, 64)
        dom[b] = int(toks[(37 * b + 11) % L])
        _plant_dominant(rows, q, dom[b], (b, 0), 5 + b)
    _clear_others(rows, dom, lambda b: 5 + b)
    case.kv_rows = rows
    case.q = q
    raw, out, _, (st, bits) = _run_dense(case, f)
    assert st == 0, (st, bits)
    want = torch.from_numpy(f["odq"](raw.cpu().numpy())).to(torch.bfloat16)
    for b, r in dom.items():
        assert torch.equal(out[b, 0].cpu(), want[r].unsqueeze(0).expand(128, 512)), b


def test_fp8_528_scale_beyond_range_is_reported():
    """The 528-byte rows are dequantised to fp16: a block amax of 6e4 needs a
    scale of 2^8, whose largest products exceed 65504: reported, not passed
    silently; 2^7 (amax 5e4) still decodes within tolerance."""
    f = FORMATS["fp8_528"]
    for amax, ok in [(5e4, True), (6e4, False)]:
        case = synth.make_dense_case([100], seed=98, d_k=512)
        case.kv_rows[3, 40] = amax
        case.q[..., 40] = 0          # keep the scores ordinary
        raw, out, lse, (st, bits) = _run_dense(case, f)
        if ok:
            assert st == 0, (st, bits)
            ro, rl = _oracle_dense(case, raw, f)
            assert_close_attn(out, lse, ro, rl, "528 scale 2^15")
        else:
            assert st == MLA_ERR_RANGE and bits & 8, (st, bits)


@pytest.mark.parametrize("name", list(FORMATS))
def test_query_beyond_fp16_is_reported(name):
    """The latent product of quantised rows runs in fp16: a bf16 query entry
    beyond 65504 is saturated and reported."""
    f = FORMATS[name]
    case = synth.make_dense_case([100, 7], seed=100, d_k=512)
    case.q[1, 0, 5, 300] = 1e5
    _, _, _, (st, bits) = _run_dense(case, f)
    assert st == MLA_ERR_RANGE and bits & 8, (st, bits)


@pytest.mark.parametrize("name", list(FORMATS))
@pytest.mark.parametrize("delta", [12, 60])
def test_split_peaks(name, delta):
    """The two CTAs of a pair sum dims [0, 256) and [256, 512) of a V4.1 key.
    Two tokens per request have partial scores delta log2 units apart in
    opposite directions (the first half's maximum on one token, the second
    half's on the other): within about 22 binades the rows are certified and
    match the oracle, beyond it they are reported. The signal is spread over
    32 dims of each half, so that the value rows stay of order 1 (the
    acceptance bound is absolute for small outputs)."""
    f = FORMATS[name]
    case = synth.make_dense_case([200, 77], seed=99, d_k=512)
    n_sig, alpha = 32, 8.0
    d0, d1 = list(range(0, n_sig)), list(range(256, 256 + n_sig))
    u = case.softmax_scale * 1.4426950408889634 * alpha * n_sig
    rows, q = case.kv_rows, case.q
    rows[:, d0 + d1] = 0
    q[..., d0 + d1] = alpha
    bt = case.block_table.numpy()
    rng = np.random.default_rng(99)
    for b, L in enumerate([200, 77]):
        toks = synth.paged_rows_index(bt[b], L, 64)
        pick = rng.choice(toks, size=2, replace=False)
        for n, r in enumerate(pick):
            x, y = (delta + 8) / 2 / u, (delta - 8) / 2 / u
            hi, lo = (d0, d1) if n == 0 else (d1, d0)
            rows[r, hi] = x
            rows[r, lo] = -y
    raw, out, lse, (st, bits) = _run_dense(case, f)
    if delta > 22:
        assert st == MLA_ERR_RANGE and bits & 8, (st, bits)
        return
    assert st == 0, (st, bits)
    ro, rl = _oracle_dense(case, raw, f)
    assert_close_attn(out, lse, ro, rl, f"{name} split peaks delta={delta}")


@pytest.mark.parametrize("name", list(FORMATS))
def test_split_and_combine_entry_points(name):
    """mla_decode_splitkv followed by mla_combine_splits equals the one-call
    decode for the V4.1 rows (requests cut into pieces by parts = 3)."""
    f = FORMATS[name]
    case = synth.make_dense_case([300, 77, 1], seed=101, d_k=512)
    raw = f["quant"](case.kv_rows.to(DEV))
    sl, bt = case.cache_seqlens.to(DEV), case.block_table.to(DEV)
    kv = raw.view(case.num_blocks, 64, 1, f["row"])
    q = case.q.to(DEV)
    meta, ns = _meta(sl, 1, f["fmt"], parts=3)
    kw = dict(softmax_scale=case.softmax_scale, kv_format=f["fmt"])
    mla.mla_read_status(device=DEV)
    o1, l1 = mla.mla_decode_with_kvcache(q, kv, bt, sl, 512, meta, ns, **kw)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    mla.mla_decode_splitkv(q, kv, bt, sl, 512, meta, ns, out=o2, lse=l2, **kw)
    mla.mla_combine_splits(q, kv, bt, sl, 512, meta, ns, out=o2, lse=l2, **kw)
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, (st, bits)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
