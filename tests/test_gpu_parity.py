"""GPU parity: libmla (through its C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import assert_close_attn

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def _status_clear(dev="cuda"):
    st, bits = mla.mla_read_status(device=dev)
    return st, bits


def run_dense(case, parts=None, causal=None, dev="cuda"):
    causal = case.causal if causal is None else causal
    q = case.q.to(dev)
    kv = case.kvcache_paged().to(dev)
    bt = case.block_table.to(dev)
    sl = case.cache_seqlens.to(dev)
    meta, ns = mla.mla_get_metadata(sl, case.s_q, case.h_q, causal=causal, num_sm_parts=parts)
    out, lse = mla.mla_decode_with_kvcache(q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                           causal=causal)
    torch.cuda.synchronize()
    return out, lse, meta


def oracle_dense(case, causal=None):
    causal = case.causal if causal is None else causal
    out, lse, _ = oracle.mla_decode(oracle.to_f64(case.q), oracle.to_f64(case.kv_rows),
                                    cache_seqlens=case.cache_seqlens.numpy(), block_table=case.block_table.numpy(),
                                    page_block=case.page_block, softmax_scale=case.softmax_scale, causal=causal)
    return out, lse


# ---------------------------------------------------------------------------
# FP8 quantiser: bit-exact
# ---------------------------------------------------------------------------
def test_quantize_bitexact_random_and_special():
    rows = synth.make_latent_rows(4096, seed=21, outlier_channels=4)
    x = rows.float()
    x[0, :128] = 0.0                        # all-zero block -> scale 1
    x[1, 128:256] = 1e-30                   # tiny block
    x[2, 256:384] = torch.linspace(-3e4, 3e4, 128)
    x[3, :] = -0.0
    x[4, 384:512] = 448.0
    x[5, :512] = torch.tensor([2.0 ** (-k % 20) for k in range(512)])
    rows = x.to(torch.bfloat16)
    ref = oracle.quantize_kv_fp8(rows)
    got = mla.mla_quantize_kv_fp8(rows.cuda()).cpu().numpy()
    mism = np.argwhere(got != ref)
    assert mism.size == 0, f"{len(mism)} bytes differ, first {mism[:5].tolist()}"


def test_quantize_bitexact_full_bf16_sweep():
    """Every bf16 bit pattern that is finite appears as a latent value once,
    next to a fixed block maximum (so every x/scale ratio class is exercised)."""
    pats = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = pats.view(torch.bfloat16).float()
    vals = vals[torch.isfinite(vals)]
    vals = vals[vals.abs() <= 1e4]
    n = (vals.numel() + 126) // 127
    buf = torch.zeros(n * 127)
    buf[:vals.numel()] = vals
    blocks = buf.view(n, 127)
    rows = torch.zeros(n, 576)
    for j in range(4):
        rows[:, 128 * j:128 * j + 127] = blocks.roll(j, 0)
        rows[:, 128 * j + 127] = 1e4 * (1 + j)
    rows[:, 512:] = blocks[:, :64]
    rows = rows.to(torch.bfloat16)
    ref = oracle.quantize_kv_fp8(rows)
    got = mla.mla_quantize_kv_fp8(rows.cuda()).cpu().numpy()
    assert (got == ref).all()


# ---------------------------------------------------------------------------
# dense BF16 decode
# ---------------------------------------------------------------------------
def test_dense_config_small():
    """B=2, s_q=1, h_q=128, lengths {256,193}, shuffled pages."""
    case = synth.make_dense_case([256, 193], seed=0)
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert _status_clear()[0] == 0
    assert_close_attn(out, lse, ro, rl, "dense small")


@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [127, 1, 64, 200], [1000, 3, 129]])
def test_dense_ragged_lengths(lens):
    case = synth.make_dense_case(lens, seed=len(lens) + lens[0])
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, f"lens={lens}")


@pytest.mark.parametrize("parts", [1, 2, 3, 7, 40])
def test_split_invariance(parts):
    """The result does not depend on how the schedule cuts the requests."""
    case = synth.make_dense_case([700, 64, 1500, 333], seed=5)
    out, lse, _ = run_dense(case, parts=parts)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, f"parts={parts}")


def test_empty_request_gives_zero_and_neg_inf():
    case = synth.make_dense_case([0, 70], seed=6)
    out, lse, _ = run_dense(case)
    o = out.float().cpu()
    assert (o[0] == 0).all() and torch.isneginf(lse[0].cpu()).all()
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, "empty + 70")


def test_masked_rows_never_leak_nan():
    """Rows beyond each length (page tails, spare pages) hold NaN."""
    case = synth.make_dense_case([65, 1, 130], seed=7, spare_blocks=2, tail_fill=float("nan"))
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, "nan tails")


def test_causal_s_q2():
    case = synth.make_dense_case([300, 64, 1], s_q=2, causal=True, seed=8)
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, "causal s_q=2")


def test_noncausal_s_q2():
    case = synth.make_dense_case([129, 40], s_q=2, causal=False, seed=9)
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, "non-causal s_q=2")


def test_fp16_cache():
    case = synth.make_dense_case([257, 90], dtype=torch.float16, seed=10)
    out, lse, _ = run_dense(case)
    ro, rl = oracle_dense(case)
    assert out.dtype == torch.float16
    assert_close_attn(out, lse, ro, rl, "fp16")


def test_gather_exact_single_dominant_key():
    """One key with a score margin of about 200 log2 units -> p = 1 and every
    other p = 0 in fp32, so the output equals that key's value row after the
    bf16 round trip. The margin sits in two RoPE dims (512+b and 544+b), so the
    key dominates every partial sum the kernel forms over a subset of the 576
    dims, and the scores stay near 200, where fp32 holds them to 2^-16 (a far
    larger margin would make the fp32 score itself inexact by more than the
    bf16 rounding of p tolerates)."""
    case = synth.make_dense_case([200, 130], seed=11)
    sl = case.cache_seqlens.numpy()
    bt = case.block_table.numpy()
    for b, tok in [(0, 137), (1, 64)]:
        row = synth.paged_rows_index(bt[b], int(sl[b]), 64)[tok]
        q = case.q[b, 0].float()
        kvr = case.kv_rows[row].float().clone()
        kvr[512:] = 0
        kvr[512 + b] = 26.0                        # only this key has large RoPE entries
        kvr[544 + b] = 26.0
        case.kv_rows[row] = kvr.to(torch.bfloat16)
        qq = q.clone()
        qq[:, 512 + b] = 64.0                      # 64 * 26 / 24 * log2(e) = 100 log2 units per dim
        qq[:, 544 + b] = 64.0
        case.q[b, 0] = qq.to(torch.bfloat16)
    out, lse, _ = run_dense(case)
    for b, tok in [(0, 137), (1, 64)]:
        row = synth.paged_rows_index(bt[b], int(sl[b]), 64)[tok]
        want = case.kv_rows[row, :512].unsqueeze(0).expand(128, 512)
        assert torch.equal(out[b, 0].cpu(), want), f"request {b}"


def test_stale_metadata_is_reported():
    case = synth.make_dense_case([300, 100], seed=12)
    dev = "cuda"
    q, kv = case.q.to(dev), case.kvcache_paged().to(dev)
    bt, sl = case.block_table.to(dev), case.cache_seqlens.to(dev)
    _status_clear()
    meta, ns = mla.mla_get_metadata(sl, 1, 128)
    sl2 = sl.clone()
    sl2[1] = 101
    mla.mla_decode_with_kvcache(q, kv, bt, sl2, 512, meta, ns)
    st, bits = _status_clear()
    assert st == 3 and bits & 4


def test_bad_page_is_reported_and_masked():
    case = synth.make_dense_case([130, 64], seed=13)
    bt = case.block_table.clone()
    bt[0, 1] = 10 ** 6                  # tokens 64..127 of request 0 unreachable
    dev = "cuda"
    _status_clear()
    meta, ns = mla.mla_get_metadata(case.cache_seqlens.to(dev), 1, 128)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(dev), case.kvcache_paged().to(dev), bt.to(dev),
                                           case.cache_seqlens.to(dev), 512, meta, ns)
    st, bits = _status_clear()
    assert st == 4 and bits & 1
    # request 1 is untouched; request 0 equals attention over its reachable tokens
    ro, rl = oracle_dense(case)
    assert_close_attn(out[1:], lse[1:], ro[1:], rl[1:], "other request")
    rows = synth.paged_rows_index(case.block_table.numpy()[0], 130, 64)
    keep = np.r_[0:64, 128:130]
    o2, l2 = oracle.attend(oracle.to_f64(case.q)[0, 0], oracle.to_f64(case.kv_rows)[rows[keep]], case.softmax_scale)
    assert_close_attn(out[0, 0], lse[0, 0], o2, l2, "masked page")


def test_schedule_covers_every_tile_once():
    lens = [4096, 12288, 1, 0, 65, 8192, 777]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for parts in [1, 5, 76, 200]:
        meta, ns = mla.mla_get_metadata(sl, 2, 128, causal=True, num_sm_parts=parts)
        m = meta.meta.cpu().numpy()
        off = ns.cpu().numpy()
        recs = m[16:16 + 8 * parts].reshape(parts, 8)
        B, s_q = len(lens), 2
        tiles = [max(0, lens[v % B] - s_q + 1 + v // B) for v in range(B * s_q)]
        tiles = [(L + 63) // 64 for L in tiles]
        seen = [np.zeros(n, int) for n in tiles]
        npieces = np.zeros(B * s_q, int)
        for r in recs:
            bv, bt_, ev, et = r[:4]
            if bv < 0:
                continue
            for v in range(bv, ev + 1):
                t0 = bt_ if v == bv else 0
                t1 = min(et if v == ev else tiles[v], tiles[v])
                if t1 > t0:
                    seen[v][t0:t1] += 1
                    npieces[v] += 1
        for v in range(B * s_q):
            assert (seen[v] == 1).all(), (parts, v)
            assert off[v + 1] - off[v] == npieces[v]


# ---------------------------------------------------------------------------
# FP8 656-byte cache: dense paged and token-sparse
# ---------------------------------------------------------------------------
def _fp8_oracle_rows(rows_bf16):
    """Oracle view of an FP8 cache: quantise (oracle) then dequantise in float64."""
    raw = oracle.quantize_kv_fp8(rows_bf16)
    return raw, oracle.dequantize_kv_fp8(raw)


@pytest.mark.parametrize("lens,s_q,causal", [([256, 193], 1, False), ([65, 1, 700], 1, False),
                                             ([300, 64], 2, True)])
def test_fp8_dense_paged(lens, s_q, causal):
    case = synth.make_dense_case(lens, s_q=s_q, causal=causal, seed=20 + len(lens), outlier_channels=4)
    dev = "cuda"
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(dev))
    raw_ref, deq = _fp8_oracle_rows(case.kv_rows)
    assert (raw.cpu().numpy() == raw_ref).all()
    kv8 = raw.view(case.num_blocks, 64, 1, 656)
    sl = case.cache_seqlens.to(dev)
    meta, ns = mla.mla_get_metadata(sl, s_q, 128, causal=causal, is_fp8=True)
    _status_clear()
    out, lse = mla.mla_decode_with_kvcache(case.q.to(dev), kv8, case.block_table.to(dev), sl, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, causal=causal, is_fp8=True)
    torch.cuda.synchronize()
    assert _status_clear()[0] == 0
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, cache_seqlens=case.cache_seqlens.numpy(),
                                  block_table=case.block_table.numpy(), softmax_scale=case.softmax_scale, causal=causal)
    assert_close_attn(out, lse, ro, rl, f"fp8 dense {lens}")


def _run_sparse(case, raw_dev, dev="cuda", parts=None):
    B = case.batch
    kv8 = raw_dev.view(-1, 64, 1, 656)
    idx = case.indices.to(dev)
    meta, ns = mla.mla_get_metadata(None, case.s_q, 128, batch=B, topk=idx.shape[-1], is_fp8=True, device=dev,
                                    num_sm_parts=parts)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(dev), kv8, None, None, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, is_fp8=True, indices=idx)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("s_q,topk,parts", [(1, 256, None), (2, 100, None), (1, 200, 3), (2, 64, 1),
                                             (48, 200, None)])
def test_fp8_sparse(s_q, topk, parts):
    case = synth.make_sparse_case(2, s_q, topk, tokens_per_request=2048, seed=30 + topk, outlier_channels=4)
    dev = "cuda"
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(dev))
    raw_ref, deq = _fp8_oracle_rows(case.kv_rows)
    assert (raw.cpu().numpy() == raw_ref).all()
    _status_clear()
    out, lse = _run_sparse(case, raw, parts=parts)
    assert _status_clear()[0] == 0
    ro, rl, bad = oracle.mla_decode(oracle.to_f64(case.q), deq, indices=case.indices.numpy(),
                                    softmax_scale=case.softmax_scale)
    assert not bad
    assert_close_attn(out, lse, ro, rl, f"fp8 sparse s_q={s_q} topk={topk}")


def test_fp8_sparse_out_of_range_index_reported_and_skipped():
    case = synth.make_sparse_case(1, 1, 128, tokens_per_request=1024, seed=41)
    idx = case.indices.clone()
    idx[0, 0, 3] = 1 << 30          # beyond the cache
    idx[0, 0, 70] = -5              # negative, not the -1 padding
    case.indices = idx
    dev = "cuda"
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(dev))
    _, deq = _fp8_oracle_rows(case.kv_rows)
    _status_clear()
    out, lse = _run_sparse(case, raw)
    st, bits = _status_clear()
    assert st == 4 and bits & 1
    ro, rl, bad = oracle.mla_decode(oracle.to_f64(case.q), deq, indices=idx.numpy(),
                                    softmax_scale=case.softmax_scale)
    assert bad
    assert_close_attn(out, lse, ro, rl, "fp8 sparse bad index")


def test_fp8_sparse_all_invalid_query():
    case = synth.make_sparse_case(2, 1, 64, tokens_per_request=512, seed=42)
    idx = case.indices.clone()
    idx[1] = -1
    case.indices = idx
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to("cuda"))
    out, lse = _run_sparse(case, raw)
    assert (out[1].float().cpu() == 0).all() and torch.isneginf(lse[1].cpu()).all()
