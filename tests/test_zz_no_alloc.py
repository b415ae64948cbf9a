"""The allocation-free decode entry point (mla_decode_with_kvcache_noalloc).

It exists for callers that cannot allocate device memory on demand (a
fixed-latency serving loop, a plug-in whose host owns all device memory): its
split-KV scratch is a fixed array inside the library instead of a caller
workspace. These checks call it through the C ABI and compare it with the
regular entry point, twice in a row, because the array keeps the previous
call's contents. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
from tests.helpers import assert_close_attn

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def _ref_and_noalloc(case, dev="cuda", parts=None):
    q = case.q.to(dev)
    kv = case.kvcache_paged().to(dev)
    bt, sl = case.block_table.to(dev), case.cache_seqlens.to(dev)
    meta, ns = mla.mla_get_metadata(sl, case.s_q, 128, causal=case.causal, num_sm_parts=parts)
    ref_o, ref_l = mla.mla_decode_with_kvcache(q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                               causal=case.causal)
    results = []
    for _ in range(2):     # the second call runs on the scratch the first left behind
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device=dev)
        o, l = mla.mla_decode_with_kvcache_noalloc(q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                                   causal=case.causal, status=status)
        torch.cuda.synchronize()
        results.append((o.clone(), l.clone(), int(status.item())))
    return (ref_o, ref_l), results


@pytest.mark.parametrize("lens,s_q,causal,parts", [([256, 193], 1, False, None), ([700, 64, 1500], 2, True, 5)])
def test_noalloc_matches_regular_entry_twice(lens, s_q, causal, parts):
    case = synth.make_dense_case(lens, s_q=s_q, causal=causal, seed=50 + len(lens))
    (ref_o, ref_l), results = _ref_and_noalloc(case, parts=parts)
    for o, l, status in results:
        assert status == 0
        assert_close_attn(o, l, ref_o.float().cpu().numpy(), ref_l.cpu().numpy(), "noalloc vs regular")


def test_noalloc_reports_device_status():
    case = synth.make_dense_case([300, 100], seed=61)
    dev = "cuda"
    sl = case.cache_seqlens.to(dev)
    meta, ns = mla.mla_get_metadata(sl, 1, 128)
    sl2 = sl.clone()
    sl2[0] = 301                      # lengths changed after the schedule was built
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mla.mla_decode_with_kvcache_noalloc(case.q.to(dev), case.kvcache_paged().to(dev), case.block_table.to(dev), sl2,
                                        512, meta, ns, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = "cuda"
    B = 200                           # (200 + parts) splits x 128 heads x 2 KB > 32 MiB
    sl = torch.full((B,), 64, dtype=torch.int32, device=dev)
    meta, ns = mla.mla_get_metadata(sl, 1, 128)
    case = synth.make_dense_case([64] * B, seed=62)
    with pytest.raises(mla.MLAError) as ei:
        mla.mla_decode_with_kvcache_noalloc(case.q.to(dev), case.kvcache_paged().to(dev), case.block_table.to(dev),
                                            sl, 512, meta, ns)
    assert ei.value.status == 1


@pytest.mark.parametrize("fmt,row", [(mla.KV_FP8_528, 528), (mla.KV_FP4_288, 288)])
def test_noalloc_v41_sparse_matches_regular_entry(fmt, row):
    """The V4.1 rows (kv_format 2 and 3), token-sparse, through both entry points."""
    dev = "cuda"
    case = synth.make_sparse_case(3, 2, 192, tokens_per_request=1024, seed=63, d_k=512)
    quant = mla.mla_quantize_kv_fp8_528 if fmt == mla.KV_FP8_528 else mla.mla_quantize_kv_fp4_288
    kv = quant(case.kv_rows.to(dev)).view(-1, 64, 1, row)
    q, idx = case.q.to(dev), case.indices.to(dev)
    meta, ns = mla.mla_get_metadata(None, 2, 128, batch=3, topk=192, kv_format=fmt, device=dev)
    ref_o, ref_l = mla.mla_decode_with_kvcache(q, kv, None, None, 512, meta, ns, softmax_scale=case.softmax_scale,
                                               kv_format=fmt, indices=idx)
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device=dev)
    o, l = mla.mla_decode_with_kvcache_noalloc(q, kv, None, None, 512, meta, ns, softmax_scale=case.softmax_scale,
                                               kv_format=fmt, indices=idx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close_attn(o, l, ref_o.float().cpu().numpy(), ref_l.cpu().numpy(), "noalloc vs regular, V4.1")
