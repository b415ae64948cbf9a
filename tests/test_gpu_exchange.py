"""GPU parity where the two halves of the score disagree.

The 128-head decode kernel splits the 576 dims of every score between the
two CTAs of a pair: one sums latent dims 0-255 and RoPE dims 512-543, the
other latent dims 256-511 and RoPE dims 544-575, and the score is the sum of
the two partial scores. Attention itself is exact ("矩阵、注意力与 GPU：拆解
DeepGEMM 与 FlashMLA", §五: FlashAttention reorders, it does not
approximate), so the result must not depend on how far the partial scores of
a token lie below each half's own maximum. These cases plant two tokens per
request whose partial scores disagree by delta log2 units: token A holds the
first half's maximum and its second-half score lies delta below the second
half's maximum, token B the other way round, and A and B win the full score
by 8 log2 units. The signal lives in the RoPE dims, which are not part of
the value, so the output stays an average of N(0,1) rows. Delta 12 and 20
stay within what the fp16 factors certify; delta 30 and 60 go beyond it, where
16-bit caches recompute the row exactly and FP8 caches report it.
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
ALPHA = 8.0                       # query weight on the two signal dims
LOG2E = 1.4426950408889634
D0, D1 = 512, 544                 # one RoPE dim in each half of the pair


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def _unit(scale):
    """log2 units of score per unit of cache value on a signal dim."""
    return scale * LOG2E * ALPHA


def plant_split_peaks(rows, q, tokens_of, delta, margin=8.0, every_token=False, seed=0):
    """Zero the signal dims everywhere, then give each request's A/B tokens
    partial scores (+x, -y) and (-y, +x) on dims D0/D1 with x + y = delta and
    x - y = margin (log2 units). With every_token, all of a request's tokens
    alternate A-type and B-type, each with its own margin. Edits rows/q in
    place (16-bit tensors)."""
    rng = np.random.default_rng(seed)
    scale = q.shape[-1] ** -0.5
    u = _unit(scale)
    rows[:, D0] = 0
    rows[:, D1] = 0
    q[..., D0] = ALPHA
    q[..., D1] = ALPHA
    for toks in tokens_of:
        toks = np.asarray(toks)
        if every_token:
            pick = toks
            margins = margin + rng.normal(0.0, 2.0, size=len(toks))
        else:
            pick = rng.choice(toks, size=2, replace=False)
            margins = np.full(2, margin)
        for n, r in enumerate(pick):
            x = (delta + margins[n]) / 2 / u
            y = (delta - margins[n]) / 2 / u
            hi, lo = (D0, D1) if n % 2 == 0 else (D1, D0)
            rows[r, hi] = x
            rows[r, lo] = -y


def half_scores(q64, rows64, scale):
    """Partial scores (log2 units) of the two halves: [h, T] each."""
    h0 = np.r_[0:256, 512:544]
    h1 = np.r_[256:512, 544:576]
    s = scale * LOG2E
    return s * q64[:, h0] @ rows64[:, h0].T, s * q64[:, h1] @ rows64[:, h1].T


def run_dense(case, parts=None):
    sl = case.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, case.s_q, 128, causal=case.causal, num_sm_parts=parts)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(DEV), case.kvcache_paged().to(DEV), case.block_table.to(DEV),
                                           sl, 512, meta, ns, softmax_scale=case.softmax_scale, causal=case.causal)
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, (st, bits)
    return out, lse


def dense_case(delta, every_token=False, dtype=torch.bfloat16, lens=(200, 77), seed=60):
    case = synth.make_dense_case(list(lens), dtype=dtype, seed=seed)
    bt = case.block_table.numpy()
    toks = [synth.paged_rows_index(bt[b], L, 64) for b, L in enumerate(lens)]
    plant_split_peaks(case.kv_rows, case.q, toks, delta, every_token=every_token, seed=seed)
    return case, toks


def oracle_dense(case):
    out, lse, _ = oracle.mla_decode(oracle.to_f64(case.q), oracle.to_f64(case.kv_rows),
                                    cache_seqlens=case.cache_seqlens.numpy(), block_table=case.block_table.numpy(),
                                    softmax_scale=case.softmax_scale)
    return out, lse


@pytest.mark.parametrize("delta", [12, 20, 30, 60])
@pytest.mark.parametrize("parts", [None, 3])
def test_split_peaks_bf16(delta, parts):
    case, toks = dense_case(delta)
    # the planted inputs do what they claim: on request 0 the two halves'
    # maxima lie on different tokens, each about delta above the other
    # half's value there
    s0, s1 = half_scores(oracle.to_f64(case.q)[0, 0], oracle.to_f64(case.kv_rows)[toks[0]], case.softmax_scale)
    a, b = s0.argmax(axis=1), s1.argmax(axis=1)
    assert (a != b).all()
    gap = s0.max(axis=1) - s0[np.arange(128), b]
    assert np.all(np.abs(gap - delta) < 6.0), gap[:4]
    out, lse = run_dense(case, parts)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, f"split peaks delta={delta} parts={parts}")


@pytest.mark.parametrize("parts", [None, 3])
def test_every_token_split(parts):
    """Every token of every request has one half far above the other, so no
    token's score is near either half's own maximum."""
    case, _ = dense_case(40, every_token=True, lens=(300, 64, 129), seed=61)
    out, lse = run_dense(case, parts)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, f"every token split parts={parts}")


@pytest.mark.parametrize("delta", [20, 60])
def test_split_peaks_fp16(delta):
    """fp16 caches carry P as fp16, whose range ends at 2^-24: the reference
    max must lie near the tile's true max, not at the sum of the halves'
    maxima."""
    case, _ = dense_case(delta, dtype=torch.float16, seed=62)
    out, lse = run_dense(case)
    ro, rl = oracle_dense(case)
    assert_close_attn(out, lse, ro, rl, f"fp16 split peaks delta={delta}")


MLA_ERR_RANGE = 7


@pytest.mark.parametrize("delta", [12, 60])
def test_split_peaks_fp8_dense(delta):
    """The RoPE dims of the 656-byte row stay bf16, so the planted signal
    survives quantisation. FP8 caches certify a row when its halves disagree
    by up to about 22 binades (delta 12: compared with the oracle on the
    dequantised cache) and report the rows beyond that (delta 60)."""
    case, _ = dense_case(delta, seed=63)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(DEV))
    deq = oracle.dequantize_kv_fp8(oracle.quantize_kv_fp8(case.kv_rows))
    sl = case.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, 1, 128, is_fp8=True)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(DEV), raw.view(case.num_blocks, 64, 1, 656),
                                           case.block_table.to(DEV), sl, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, is_fp8=True)
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    if delta > 22:
        assert st == MLA_ERR_RANGE and bits & 8, (st, bits)
        return
    assert st == 0, (st, bits)
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, cache_seqlens=case.cache_seqlens.numpy(),
                                  block_table=case.block_table.numpy(), softmax_scale=case.softmax_scale)
    assert_close_attn(out, lse, ro, rl, f"fp8 dense split peaks delta={delta}")


@pytest.mark.parametrize("delta", [12, 60])
def test_split_peaks_fp8_sparse(delta):
    case = synth.make_sparse_case(2, 2, 192, tokens_per_request=1024, seed=64)
    idx = case.indices.numpy()
    toks = [idx[b, i][idx[b, i] >= 0] for b in range(2) for i in range(2)]
    plant_split_peaks(case.kv_rows, case.q, toks, delta, seed=64)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows.to(DEV))
    deq = oracle.dequantize_kv_fp8(oracle.quantize_kv_fp8(case.kv_rows))
    meta, ns = mla.mla_get_metadata(None, 2, 128, batch=2, topk=192, is_fp8=True, device=DEV)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q.to(DEV), raw.view(-1, 64, 1, 656), None, None, 512, meta, ns,
                                           softmax_scale=case.softmax_scale, is_fp8=True,
                                           indices=case.indices.to(DEV))
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    if delta > 22:
        assert st == MLA_ERR_RANGE and bits & 8, (st, bits)
        return
    assert st == 0, (st, bits)
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), deq, indices=idx, softmax_scale=case.softmax_scale)
    assert_close_attn(out, lse, ro, rl, f"fp8 sparse split peaks delta={delta}")
