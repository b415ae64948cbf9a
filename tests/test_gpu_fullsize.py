"""GPU parity at the benchmark's full sizes, on sampled outputs.

Each test builds one of the benchmark's workloads at its full size, runs the
decode once over the whole batch in the launch configuration the benchmark
times (default split-KV schedule, one call), and recomputes a few sampled
(request, query position) rows -- all 128 heads each -- with the float64
oracle. FP8 caches are quantised on the CPU by the oracle for the sampled
requests; those bytes are checked to equal the library's cache (the quantiser
is bit-exact), and the oracle attends over their dequantised values.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import assert_close_attn

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")
bench = pytest.importorskip("bench")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


DEV = "cuda"


def _run(w, case, kv, bt, sl, idx):
    s_q = w["s_q"]
    is_fp8 = w["kind"] != "dense"
    if w["kind"] == "sparse":
        meta, ns = mla.mla_get_metadata(None, s_q, 128, batch=case.batch, topk=idx.shape[-1], is_fp8=True,
                                        device=DEV)
    else:
        meta, ns = mla.mla_get_metadata(sl, s_q, 128, causal=w["causal"], is_fp8=is_fp8)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                           causal=w["causal"], is_fp8=is_fp8, indices=idx)
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, f"device status {st} bits {bits}"
    return out, lse


def _samples(B, s_q, n=4, seed=7):
    """A few requests (first, last, random), and for each every query position
    when s_q is small, else the first, the last and two random ones."""
    rng = np.random.default_rng(seed)
    bs = sorted(set([0, B - 1] + [int(x) for x in rng.integers(0, B, size=n - 2)]))
    out = []
    for b in bs:
        qs = range(s_q) if s_q <= 4 else sorted(set([0, s_q - 1] + [int(x) for x in rng.integers(0, s_q, size=2)]))
        out += [(b, i) for i in qs]
    return out


@pytest.mark.parametrize("workload", ["dense_bf16_b64_sq1_l8192", "dense_bf16_b64_sq1_uniform",
                                      "dense_bf16_b64_sq2_causal_uniform"])
def test_dense_bf16_full_size_sampled(workload):
    w = bench.WORKLOADS[workload]
    case, seqlens = bench.build_case(w, DEV)
    bt, sl = case.block_table.to(DEV), case.cache_seqlens.to(DEV)
    out, lse = _run(w, case, case.kvcache_paged(), bt, sl, None)
    bt_np = case.block_table.numpy()
    for b, i in _samples(case.batch, w["s_q"]):
        L = int(seqlens[b]) - (w["s_q"] - 1 - i if w["causal"] else 0)
        rows = synth.paged_rows_index(bt_np[b], L, case.page_block)
        keys = oracle.to_f64(case.kv_rows[torch.from_numpy(rows).to(DEV)].cpu())
        ro, rl = oracle.attend(oracle.to_f64(case.q[b, i].cpu()), keys, case.softmax_scale)
        assert_close_attn(out[b, i], lse[b, i], ro, rl, f"{workload} b={b} i={i}")


def test_fp8_dense_full_size_sampled():
    w = bench.WORKLOADS["fp8_dense_b16_l32768"]
    case, seqlens = bench.build_case(w, DEV)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows)
    bt, sl = case.block_table.to(DEV), case.cache_seqlens.to(DEV)
    out, lse = _run(w, case, raw.view(case.num_blocks, 64, 1, 656), bt, sl, None)
    bt_np = case.block_table.numpy()
    for b, i in _samples(case.batch, 1, n=3):
        rows = synth.paged_rows_index(bt_np[b], int(seqlens[b]), case.page_block)
        ridx = torch.from_numpy(rows).to(DEV)
        raw_ref = oracle.quantize_kv_fp8(case.kv_rows[ridx].cpu())
        assert (raw[ridx].cpu().numpy() == raw_ref).all(), "quantised rows differ"
        ro, rl = oracle.attend(oracle.to_f64(case.q[b, i].cpu()), oracle.dequantize_kv_fp8(raw_ref),
                               case.softmax_scale)
        assert_close_attn(out[b, i], lse[b, i], ro, rl, f"fp8 dense b={b}")


@pytest.mark.parametrize("workload", ["fp8_sparse_b32_sq2_topk32768", "fp8_sparse_b32_sq1_topk2048",
                                      "fp8_sparse_prefill_b4_sq1024_topk2048"])
def test_fp8_sparse_full_size_sampled(workload):
    w = bench.WORKLOADS[workload]
    case, _ = bench.build_case(w, DEV)
    raw = mla.mla_quantize_kv_fp8(case.kv_rows)
    idx = case.indices.to(DEV)
    out, lse = _run(w, case, raw.view(-1, 64, 1, 656), None, None, idx)
    idx_np = case.indices.numpy()
    for b, i in _samples(case.batch, w["s_q"], n=3):
        sel = idx_np[b, i]
        sel = sel[sel != -1].astype(np.int64)
        ridx = torch.from_numpy(sel).to(DEV)
        raw_ref = oracle.quantize_kv_fp8(case.kv_rows[ridx].cpu())
        assert (raw[ridx].cpu().numpy() == raw_ref).all(), "quantised rows differ"
        ro, rl = oracle.attend(oracle.to_f64(case.q[b, i].cpu()), oracle.dequantize_kv_fp8(raw_ref),
                               case.softmax_scale)
        assert_close_attn(out[b, i], lse[b, i], ro, rl, f"{workload} b={b} i={i}")


@pytest.mark.parametrize("workload", ["v41_fp8_dense_b16_l32768", "v41_fp4_dense_b16_l32768",
                                      "v41_fp8_sparse_b32_sq1_topk32768", "v41_fp4_sparse_b32_sq1_topk32768",
                                      "v41_fp8_sparse_b32_sq1_topk2048", "v41_fp4_sparse_b32_sq1_topk2048"])
def test_v41_full_size_sampled(workload):
    """The V4.1 rows of 512 values (528-byte FP8, 288-byte FP4) at the
    benchmark's sizes: the library's rows of the sampled requests equal the
    oracle's quantisation byte for byte, and the oracle attends over their
    dequantised values."""
    w = bench.WORKLOADS[workload]
    fmt, row_bytes, d_k, qname, dqname = bench.FORMATS[bench.workload_format(w)]
    oq = getattr(oracle, qname[len("mla_"):])          # mla_quantize_kv_* -> quantize_kv_*
    odq = getattr(oracle, dqname)
    case, seqlens = bench.build_case(w, DEV)
    raw = getattr(mla, qname)(case.kv_rows)
    if w["kind"] == "sparse":
        idx = case.indices.to(DEV)
        meta, ns = mla.mla_get_metadata(None, 1, 128, batch=case.batch, topk=idx.shape[-1], kv_format=fmt,
                                        device=DEV)
        kv, bt, sl = raw.view(-1, 64, 1, row_bytes), None, None
    else:
        idx = None
        bt, sl = case.block_table.to(DEV), case.cache_seqlens.to(DEV)
        meta, ns = mla.mla_get_metadata(sl, 1, 128, kv_format=fmt)
        kv = raw.view(case.num_blocks, 64, 1, row_bytes)
    mla.mla_read_status(device=DEV)
    out, lse = mla.mla_decode_with_kvcache(case.q, kv, bt, sl, 512, meta, ns, softmax_scale=case.softmax_scale,
                                           kv_format=fmt, indices=idx)
    torch.cuda.synchronize()
    st, bits = mla.mla_read_status(device=DEV)
    assert st == 0, f"device status {st} bits {bits}"
    assert case.q.shape[-1] == d_k == 512
    for b, i in _samples(case.batch, 1, n=3):
        if idx is not None:
            sel = case.indices.numpy()[b, i]
            rows = sel[sel != -1].astype(np.int64)
        else:
            rows = synth.paged_rows_index(case.block_table.numpy()[b], int(seqlens[b]), case.page_block)
        ridx = torch.from_numpy(rows).to(DEV)
        raw_ref = oq(case.kv_rows[ridx].cpu())
        assert (raw[ridx].cpu().numpy() == raw_ref).all(), "quantised rows differ"
        ro, rl = oracle.attend(oracle.to_f64(case.q[b, i].cpu()), odq(raw_ref), case.softmax_scale)
        assert_close_attn(out[b, i], lse[b, i], ro, rl, f"{workload} b={b} i={i}")
