"""GPU parity of the few-heads (h_q = 16) decode against the float64 oracle.

The kernel computes the same attention as the 128-head path through the
transposed formulation of the FlashMLA-ETAP page (§2.2, §3.2): tokens fill
the MMA's M dimension and the 16 heads its N dimension. Shapes follow the
ETAP-shaped workload: fp16 query and cache, h_q = 16, d_qk = 576, d_v = 512.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import assert_close_attn

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")

H = 16
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def run(case, parts=None):
    q = case.q.to(DEV)
    kv = case.kvcache_paged().to(DEV)
    bt, sl = case.block_table.to(DEV), case.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, case.s_q, H, causal=case.causal, num_sm_parts=parts)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                           causal=case.causal)
    torch.cuda.synchronize()
    return out, lse


def ref(case):
    ro, rl, _ = oracle.mla_decode(oracle.to_f64(case.q), oracle.to_f64(case.kv_rows),
                                  cache_seqlens=case.cache_seqlens.numpy(), block_table=case.block_table.numpy(),
                                  softmax_scale=case.softmax_scale, causal=case.causal)
    return ro, rl


def test_default_parts_is_one_cta_per_sm():
    n = mla.mla_num_sm_parts(DEV, H)
    assert n >= torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_fewheads_small(dtype):
    case = synth.make_dense_case([256, 193], h_q=H, dtype=dtype, seed=70)
    out, lse = run(case)
    assert mla.mla_read_status(device=DEV)[0] == 0
    assert out.dtype == dtype
    assert_close_attn(out, lse, *ref(case), f"h16 small {dtype}")


@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [1000, 3, 129], [0, 70]])
def test_fewheads_ragged_and_empty(lens):
    case = synth.make_dense_case(lens, h_q=H, dtype=torch.float16, seed=71 + len(lens))
    out, lse = run(case)
    assert_close_attn(out, lse, *ref(case), f"h16 lens={lens}")


@pytest.mark.parametrize("parts", [1, 3, 40])
def test_fewheads_split_invariance(parts):
    case = synth.make_dense_case([700, 64, 1500, 333], h_q=H, dtype=torch.float16, seed=75)
    out, lse = run(case, parts=parts)
    assert_close_attn(out, lse, *ref(case), f"h16 parts={parts}")


@pytest.mark.parametrize("parts", [2, 5, 9])
def test_fewheads_many_short_pieces(parts):
    """Several pieces per CTA, among them empty requests and pieces of one to
    three tiles that follow longer ones (the producer runs ahead across piece
    boundaries, the query slot turns over every piece)."""
    case = synth.make_dense_case([0, 70, 1, 200, 0, 129, 64, 3, 1100, 2], s_q=2, causal=True, h_q=H,
                                 dtype=torch.float16, seed=79)
    out, lse = run(case, parts=parts)
    assert mla.mla_read_status(device=DEV)[0] == 0
    assert_close_attn(out, lse, *ref(case), f"h16 short pieces parts={parts}")


def test_fewheads_causal_s_q2_and_nan_tails():
    case = synth.make_dense_case([300, 64, 1], s_q=2, causal=True, h_q=H, dtype=torch.float16, seed=76,
                                 spare_blocks=2, tail_fill=float("nan"))
    out, lse = run(case)
    assert_close_attn(out, lse, *ref(case), "h16 causal s_q=2, NaN tails")


def test_fewheads_stale_metadata_is_reported():
    case = synth.make_dense_case([300, 100], h_q=H, dtype=torch.float16, seed=77)
    sl = case.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, 1, H)
    sl2 = sl.clone()
    sl2[1] = 101
    mla.mla_read_status(device=DEV)
    mla.mla_decode_with_kvcache(case.q.to(DEV), case.kvcache_paged().to(DEV), case.block_table.to(DEV), sl2, 512,
                                meta, ns)
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 3 and bits & 4


@pytest.mark.parametrize("B,L", [(16, 65536), (32, 512)])
def test_fewheads_full_size_sampled(B, L):
    """The ETAP-shaped workload at full size (identity block table, as the
    pages do not page it), compared on sampled requests."""
    case = synth.make_dense_case([L] * B, h_q=H, dtype=torch.float16, seed=78, shuffle=False, device=DEV)
    bt, sl = case.block_table.to(DEV), case.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, 1, H)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q, case.kvcache_paged(), bt, sl, 512, meta, ns,
                                           softmax_scale=case.softmax_scale)
    torch.cuda.synchronize()
    assert mla.mla_read_status(device=DEV)[0] == 0
    bt_np = case.block_table.numpy()
    for b in sorted({0, B // 2, B - 1}):
        rows = synth.paged_rows_index(bt_np[b], L, 64)
        keys = oracle.to_f64(case.kv_rows[torch.from_numpy(rows).to(DEV)].cpu())
        ro, rl = oracle.attend(oracle.to_f64(case.q[b, 0].cpu()), keys, case.softmax_scale)
        assert_close_attn(out[b, 0], lse[b, 0], ro, rl, f"h16 B={B} L={L} b={b}")


def test_fewheads_rejects_fp8_and_sparse():
    sl = torch.full((2,), 64, dtype=torch.int32, device=DEV)
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_get_metadata(sl, 1, H, is_fp8=True)
    assert ei.value.status == 2
