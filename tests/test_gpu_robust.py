"""GPU checks at the edges: exact gathering from FP8 caches, the fp16 range
of the FP8 path, and a device wait that runs out.

* Gathering is exact ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §八: a
  sparse index is an absolute cache row, -1 a padding slot; "FlashMLA 实战",
  §最小调用: block_table maps a request's pages). With one key dominating
  every other by about 200 log2 units, p = 1 for it and 0 for the rest, so the
  output must equal that key's dequantised value row bit for bit. Every block
  of the rows has amax 7 = 448 * 2^-6, so the block scale is 2^-6 and every
  dequantised value (an e4m3 code times 2^-6) is exact in fp16 and in bf16.
* The FP8 path computes the latent product in fp16 ("FlashMLA 实战", §FP8 缓存
  怎么把 KV 压掉四成: e4m3 values with one fp32 scale per 128): blocks with a
  tiny amax still meet the acceptance bound, and a query or block scale beyond
  fp16's range is reported as MLA_ERR_RANGE rather than passed silently.
* The time-out path: a test hook makes every CTA wait on a barrier nothing
  arrives at, before anything is issued; the wait gives up, the status word
  says so, and the next call on the same context is correct again.
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
MLA_ERR_TIMEOUT, MLA_ERR_RANGE = 5, 7


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def exact_fp8_rows(n, seed):
    """bf16 rows whose every latent block has amax exactly 7 (scale 2^-6)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 576, generator=g).clamp(-6.5, 6.5)
    sign = torch.where(torch.rand(n, 4, generator=g) < 0.5, -1.0, 1.0)
    for j in range(4):
        x[:, 128 * j + (7 * j) % 128] = 7.0 * sign[:, j]
    return x.to(torch.bfloat16)


def dequantised_bf16(raw):
    """The oracle's dequantised latent values of FP8 rows as bf16, checked to
    be exact in bf16 (which holds for rows from exact_fp8_rows)."""
    deq = oracle.dequantize_kv_fp8(raw.cpu().numpy())[:, :512]
    b16 = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(b16.double().numpy(), deq), "dequantised values not exact in bf16"
    return b16


def plant_dominant(rows, q, row, qi, c):
    """Make cache row `row` dominate query position qi (all heads) through
    RoPE dims 512+c and 544+c: 64 * 26 / 24 * log2(e) = 100 log2 units each."""
    rows[row, 512 + c] = 26.0
    rows[row, 544 + c] = 26.0
    q[qi][..., 512 + c] = 64.0
    q[qi][..., 544 + c] = 64.0


def _fp8_decode(q, raw, *, bt=None, sl=None, idx=None, s_q=1, causal=False):
    if idx is not None:
        meta, ns = mla.mla_get_metadata(None, s_q, 128, batch=q.shape[0], topk=idx.shape[-1], is_fp8=True,
                                        device=DEV)
    else:
        meta, ns = mla.mla_get_metadata(sl, s_q, 128, causal=causal, is_fp8=True)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(q, raw.view(-1, 64, 1, 656), bt, sl, 512, meta, ns, is_fp8=True,
                                           indices=idx, causal=causal)
    torch.cuda.synchronize()
    return out, lse, mla.mla_read_status(device=DEV)


def test_fp8_sparse_gather_exact():
    """Indices scattered over the whole cache (every request may name any
    row), -1 padding, s_q = 2: each query position's output is its dominant
    row's dequantised value, bit for bit."""
    B, s_q, topk, nrows = 3, 2, 96, 4096
    rows = exact_fp8_rows(nrows, seed=70)
    rows[:, 512:] = 0
    rng = np.random.default_rng(71)
    idx = np.stack([np.stack([rng.choice(nrows, size=topk, replace=False) for _ in range(s_q)]) for _ in range(B)])
    idx = idx.astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    q = (torch.randn(B, s_q, 128, 576, generator=torch.Generator().manual_seed(72)) * 0.5).to(torch.bfloat16)
    q[..., 512:] = 0
    dom = {}
    for b in range(B):
        for i in range(s_q):
            valid = np.flatnonzero(idx[b, i] >= 0)
            r = int(idx[b, i, rng.choice(valid)])
            c = (b * s_q + i) % 32
            plant_dominant(rows, q, r, (b, i), c)
            dom[(b, i)] = r
    # a dominant row of one query must not dominate another query too
    assert len(set(dom.values())) == len(dom)
    raw = mla.mla_quantize_kv_fp8(rows.to(DEV))
    want = dequantised_bf16(raw)
    out, lse, (st, bits) = _fp8_decode(q.to(DEV), raw, idx=torch.from_numpy(idx).to(DEV), s_q=s_q)
    assert st == 0, (st, bits)
    for (b, i), r in dom.items():
        assert torch.equal(out[b, i].cpu(), want[r].unsqueeze(0).expand(128, 512)), (b, i)


def test_fp8_paged_gather_exact():
    """The same through a shuffled block table (dense FP8 decode)."""
    case = synth.make_dense_case([200, 130, 64], seed=73)
    rows = exact_fp8_rows(case.kv_rows.shape[0], seed=74)
    rows[:, 512:] = 0
    q = torch.zeros_like(case.q)
    q[..., :512] = (case.q[..., :512].float() * 0.5).to(torch.bfloat16)
    bt, sl = case.block_table.numpy(), case.cache_seqlens.numpy()
    dom = {}
    for b, tok in [(0, 137), (1, 64), (2, 0)]:
        r = int(synth.paged_rows_index(bt[b], int(sl[b]), 64)[tok])
        plant_dominant(rows, q, r, (b, 0), b)
        dom[b] = r
    raw = mla.mla_quantize_kv_fp8(rows.to(DEV))
    want = dequantised_bf16(raw)
    out, lse, (st, bits) = _fp8_decode(q.to(DEV), raw, bt=case.block_table.to(DEV), sl=case.cache_seqlens.to(DEV))
    assert st == 0, (st, bits)
    for b, r in dom.items():
        assert torch.equal(out[b, 0].cpu(), want[r].unsqueeze(0).expand(128, 512)), b


@pytest.mark.parametrize("amax", [1e-2, 1e-4, 1e-6])
def test_fp8_small_blocks(amax):
    """Latent blocks with a tiny amax: the block scale amax/448 is an fp16
    subnormal (or flushes to zero at 1e-6), so each dequantised value carries
    an absolute error of at most 2^-15; with N(0,1) queries the result still
    meets the acceptance bound against the oracle on the exact dequantised
    cache. Half of the rows are small, half N(0,1), in every request."""
    case = synth.make_dense_case([300, 129], seed=75, outlier_channels=4)
    rows = case.kv_rows.float()
    small = torch.zeros(rows.shape[0], dtype=torch.bool)
    small[::2] = True
    blk = rows[small, :512].view(-1, 4, 128)
    blk = blk / blk.abs().amax(dim=2, keepdim=True) * amax
    rows[small, :512] = blk.view(-1, 512)
    case.kv_rows = rows.to(torch.bfloat16)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(DEV))
    deq = oracle.dequantize_kv_fp8(oracle.quantize_kv_fp8(case.kv_rows))
    out, lse, (st, bits) = _fp8_decode(case.q.to(DEV), raw, bt=case.block_table.to(DEV),
                                       sl=case.cache_seqlens.to(DEV))
    assert st == 0, (st, bits)
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, cache_seqlens=case.cache_seqlens.numpy(),
                                  block_table=case.block_table.numpy(), softmax_scale=case.softmax_scale)
    assert_close_attn(out, lse, ro, rl, f"fp8 small blocks amax={amax}")


def test_fp8_query_beyond_fp16_is_reported():
    case = synth.make_dense_case([100], seed=76)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(DEV))
    q = case.q.clone()
    q[0, 0, 5, 17] = 1.0e5                      # bf16 holds it, fp16 does not
    _, _, (st, bits) = _fp8_decode(q.to(DEV), raw, bt=case.block_table.to(DEV), sl=case.cache_seqlens.to(DEV))
    assert st == MLA_ERR_RANGE and bits & 8, (st, bits)
    # in range again: no report
    _, _, (st, bits) = _fp8_decode(case.q.to(DEV), raw, bt=case.block_table.to(DEV), sl=case.cache_seqlens.to(DEV))
    assert st == 0, (st, bits)


@pytest.mark.parametrize("sparse", [False, True])
def test_fp8_block_scale_beyond_fp16_is_reported(sparse):
    case = synth.make_dense_case([100], seed=77)
    rows = case.kv_rows.clone()
    vis = synth.paged_rows_index(case.block_table.numpy()[0], 100, 64)
    rows[int(vis[10]), 130] = 7.0e4             # block amax above 65408
    raw = mla.mla_quantize_kv_fp8(rows.to(DEV))
    if sparse:
        idx = torch.from_numpy(vis[None, None, :96].astype(np.int32)).to(DEV)
        _, _, (st, bits) = _fp8_decode(case.q.to(DEV), raw, idx=idx)
    else:
        _, _, (st, bits) = _fp8_decode(case.q.to(DEV), raw, bt=case.block_table.to(DEV),
                                       sl=case.cache_seqlens.to(DEV))
    assert st == MLA_ERR_RANGE and bits & 8, (st, bits)


# ---------------------------------------------------------------------------
# a device wait that runs out
# ---------------------------------------------------------------------------
STALL = 2_000_000      # SM cycles: about a millisecond


@pytest.fixture
def stall():
    mla.mla_set_test_stall(STALL)
    try:
        yield
    finally:
        mla.mla_set_test_stall(0)


def _dense(case, dev=DEV):
    sl = case.cache_seqlens.to(dev)
    meta, ns = mla.mla_get_metadata(sl, case.s_q, case.h_q)
    return mla.mla_decode_with_kvcache(case.q.to(dev), case.kvcache_paged().to(dev), case.block_table.to(dev), sl,
                                       512, meta, ns, softmax_scale=case.softmax_scale)


@pytest.mark.parametrize("h_q,dtype", [(128, torch.bfloat16), (16, torch.float16)])
def test_decode_wait_timeout_is_reported(h_q, dtype):
    case = synth.make_dense_case([256, 193], h_q=h_q, dtype=dtype, seed=80, shuffle=h_q == 128)
    mla.mla_read_status(device=DEV)
    mla.mla_set_test_stall(STALL)
    try:
        _dense(case)
        st, bits = mla.mla_read_status(device=DEV)
    finally:
        mla.mla_set_test_stall(0)
    assert st == MLA_ERR_TIMEOUT and bits & 2, (st, bits)
    # the context is still usable and the next call is correct
    out, lse = _dense(case)
    assert mla.mla_read_status(device=DEV)[0] == 0
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), oracle.to_f64(case.kv_rows),
                                  cache_seqlens=case.cache_seqlens.numpy(), block_table=case.block_table.numpy(),
                                  softmax_scale=case.softmax_scale)
    assert_close_attn(out, lse, ro, rl, f"after time-out h_q={h_q}")


def test_absorb_wait_timeout_is_reported():
    case = synth.make_absorb_case(5, h=3, seed=81)
    status = torch.zeros(64, dtype=torch.int32, device=DEV)
    q_out = torch.zeros(5, 3, 576, dtype=torch.bfloat16, device=DEV)
    mla.mla_set_test_stall(STALL)
    try:
        mla.mla_absorb_q(case.q_nope.to(DEV), case.w_uk.to(DEV), q_out, status=status)
        st, bits = mla.mla_read_status(status, device=DEV)
        assert st == MLA_ERR_TIMEOUT and bits & 2, (st, bits)
        mla.mla_up_project(case.o_lat.to(DEV), case.w_uv.to(DEV), status=status)
        st, bits = mla.mla_read_status(status, device=DEV)
        assert st == MLA_ERR_TIMEOUT and bits & 2, (st, bits)
    finally:
        mla.mla_set_test_stall(0)
    o = mla.mla_up_project(case.o_lat.to(DEV), case.w_uv.to(DEV), status=status)
    assert mla.mla_read_status(status, device=DEV)[0] == 0
    ref = oracle.up_project(oracle.to_f64(case.o_lat), oracle.to_f64(case.w_uv))
    assert np.abs(o.float().cpu().numpy() - ref).max() <= 8e-3 + 1e-2 * np.abs(ref).max()
