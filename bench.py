#!/usr/bin/env python
"""Benchmark of MLA decode over a paged latent KV cache on GB300.

Default workload (the headline): dense BF16 cache, B=64 requests, s_q=1,
h_q=128 heads x 576 (512 latent + 64 RoPE), every request 8192 tokens,
64-token pages in a seeded shuffled block table. One step = one pass of the
hot path: split-KV schedule (mla_get_metadata) + decode (split kernel +
combine) over the whole batch.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload NAME]

Prints ONE JSON line (rank 0). Under torchrun with N > 1 every rank runs an
independent replica of the workload on its own GPU (weak scaling, no
collective on the data path); the timed region is bracketed by a barrier and
a device synchronisation and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOPS + KV GB/s (fraction of GB300 roofline), B=64 s_q=1 seqlen 8K"

WORKLOADS = {
    # dense BF16 paged cache (the headline is the first)
    "dense_bf16_b64_sq1_l8192": dict(kind="dense", batch=64, s_q=1, lens=("fixed", 8192), causal=False),
    "dense_bf16_b64_sq1_uniform": dict(kind="dense", batch=64, s_q=1, lens=("uniform", 4096, 12288), causal=False),
    "dense_bf16_b64_sq2_causal_l8192": dict(kind="dense", batch=64, s_q=2, lens=("fixed", 8192), causal=True),
    "dense_bf16_b64_sq2_causal_uniform": dict(kind="dense", batch=64, s_q=2, lens=("uniform", 4096, 12288),
                                              causal=True),
    # 656-byte FP8 cache, paged, per-row outlier channels x8
    "fp8_dense_b16_l32768": dict(kind="fp8", batch=16, s_q=1, lens=("fixed", 32768), causal=False),
    # few heads (h_q=16, fp16, identity block table): the transposed kernel,
    # B in {16, 32} over lengths 512 .. 64K (below, added in a loop); a cache
    # smaller than twice the 129 MB L2 is one of several block-table sets that
    # the steps rotate through: a rotation reads at least twice the L2, and at
    # least the L2 passes between two uses of one set
    # token-sparse over a 131072-token FP8 cache per request, 5% of the slots -1
    "fp8_sparse_b32_sq1_topk2048": dict(kind="sparse", batch=32, s_q=1, topk=2048, causal=False),
    "fp8_sparse_b32_sq1_topk32768": dict(kind="sparse", batch=32, s_q=1, topk=32768, causal=False),
    "fp8_sparse_b32_sq2_topk2048": dict(kind="sparse", batch=32, s_q=2, topk=2048, causal=False),
    "fp8_sparse_b32_sq2_topk32768": dict(kind="sparse", batch=32, s_q=2, topk=32768, causal=False),
    # sparse prefill: 1024 query tokens per request, each with its own top-2048 list
    "fp8_sparse_prefill_b4_sq1024_topk2048": dict(kind="sparse", batch=4, s_q=1024, topk=2048, causal=False),
    # V4.1 rows of 512 values (d_k = d_v = 512): 528-byte FP8 (e4m3 + UE8M0 per
    # 32) and 288-byte FP4 (e2m1 + e4m3 per 16), token-sparse and paged
    "v41_fp8_sparse_b32_sq1_topk2048": dict(kind="sparse", batch=32, s_q=1, topk=2048, causal=False, fmt="fp8_528"),
    "v41_fp8_sparse_b32_sq1_topk32768": dict(kind="sparse", batch=32, s_q=1, topk=32768, causal=False,
                                             fmt="fp8_528"),
    "v41_fp4_sparse_b32_sq1_topk2048": dict(kind="sparse", batch=32, s_q=1, topk=2048, causal=False, fmt="fp4_288"),
    "v41_fp4_sparse_b32_sq1_topk32768": dict(kind="sparse", batch=32, s_q=1, topk=32768, causal=False,
                                             fmt="fp4_288"),
    "v41_fp8_dense_b16_l32768": dict(kind="fp8", batch=16, s_q=1, lens=("fixed", 32768), causal=False, fmt="fp8_528"),
    "v41_fp4_dense_b16_l32768": dict(kind="fp8", batch=16, s_q=1, lens=("fixed", 32768), causal=False, fmt="fp4_288"),
    # the per-head GEMMs around the kernel (q~ = W^UK^T q^C, o = W^UV o~) for the
    # headline's 64 query tokens x 128 heads; L2 flushed before every step
    "absorb_bf16_t64_h128": dict(kind="absorb", batch=64, s_q=1, h_q=128, causal=False),
}
for _b in (16, 32):
    for _l in (512, 1024, 2048, 4096, 8192, 16384, 32768, 65536):
        WORKLOADS[f"fewheads_fp16_h16_b{_b}_l{_l}"] = dict(kind="few", batch=_b, s_q=1, lens=("fixed", _l),
                                                          causal=False, h_q=16)
SPARSE_TOKENS = 131072
DEFAULT_WORKLOAD = "dense_bf16_b64_sq1_l8192"
L2_BYTES = 129e6       # GB300 L2; a workload whose touched bytes per step are below
                       # twice this rotates several index sets between steps


# cache row formats: kv_format code, bytes per row, query/key width, library
# quantiser, oracle dequantiser
FORMATS = {
    "bf16": (0, 1152, 576, None, None),
    "fp16": (0, 1152, 576, None, None),
    "fp8_656": (1, 656, 576, "mla_quantize_kv_fp8", "dequantize_kv_fp8"),
    "fp8_528": (2, 528, 512, "mla_quantize_kv_fp8_528", "dequantize_kv_fp8_528"),
    "fp4_288": (3, 288, 512, "mla_quantize_kv_fp4_288", "dequantize_kv_fp4_288"),
}


def workload_format(w) -> str:
    return w.get("fmt") or {"dense": "bf16", "few": "fp16"}.get(w["kind"], "fp8_656")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def workload_seqlens(w):
    import synth
    if w["kind"] == "sparse":
        return None
    if w["lens"][0] == "fixed":
        return [w["lens"][1]] * w["batch"]
    return [int(x) for x in synth.uniform_seqlens(w["batch"], w["lens"][1], w["lens"][2], seed=2)]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def kernel_source_digest() -> str:
    """Digest of the CUDA sources the kernels are built from (so a stored
    DRAM-traffic figure is used only for the kernels it was measured on)."""
    import hashlib
    csrc = os.path.join(ROOT, "mla_latent_kv_14_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the dominant kernel from one
    ncu capture, as recorded in profiles/dram_traffic.txt, or None when there
    is no record for this workload or the kernels changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    digest = kernel_source_digest()
    for parts in lines:
        if len(parts) >= 3 and parts[0] == workload and parts[2] == digest:
            return int(parts[1])
    return None


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of `x` over all ranks (the slowest rank's time);
    `x` itself on a single process. Works on any process-group backend
    (NCCL with a CUDA device, gloo with the CPU)."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput under weak scaling: every rank processed
    `units_per_rank` in at most `seconds` (the max over ranks)."""
    return world * units_per_rank / seconds


def work_counts(seqlens, s_q, causal, h_q=128, row_bytes=1152, indices=None, d_k=576):
    """Algorithmic FLOPs and bytes of one step (no partials, no expansion):
    FLOPs = 2 * h_q * (d_k + 512) per visible (query, key) pair; bytes = the
    cache rows read once (1152 B bf16, 656 / 528 / 288 B quantised; a row
    shared by the query positions of one request counts once) + q + out + lse
    + block table or index list."""
    if indices is not None:
        import numpy as np
        B = indices.shape[0]
        valid = indices >= 0
        pairs = int(valid.sum())
        rows = sum(len(np.unique(indices[b][valid[b]])) for b in range(B))
        kv = rows * row_bytes
        meta = indices.size * 4
    else:
        B = len(seqlens)
        pairs = 0
        for L in seqlens:
            for i in range(s_q):
                pairs += max(0, L - (s_q - 1 - i if causal else 0))
        kv = sum(seqlens) * row_bytes
        meta = sum((L + 63) // 64 for L in seqlens) * 4 + B * 4
    flops = 2.0 * h_q * (d_k + 512) * pairs
    qb = B * s_q * h_q * d_k * 2
    ob = B * s_q * h_q * (512 * 2 + 4)
    return flops, kv + qb + ob + meta, kv


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def build_case(w, device):
    import synth
    d_k = FORMATS[workload_format(w)][2]
    if w["kind"] == "sparse":
        case = synth.make_sparse_case(w["batch"], w["s_q"], w["topk"], tokens_per_request=SPARSE_TOKENS, seed=0,
                                      outlier_channels=4, device=device, d_k=d_k)
        return case, None
    seqlens = workload_seqlens(w)
    if w["kind"] == "few":
        # requests of block-table set k are k*B .. k*B+B-1 (see few_table_sets)
        case = synth.make_dense_case(seqlens * few_table_sets(seqlens), s_q=w["s_q"], h_q=w["h_q"],
                                     dtype=torch_dtype("float16"), causal=w["causal"], seed=0, device=device,
                                     shuffle=False)
        return case, seqlens
    case = synth.make_dense_case(seqlens, s_q=w["s_q"], h_q=128, causal=w["causal"], seed=0, device=device,
                                 outlier_channels=4 if w["kind"] == "fp8" else 0, d_k=d_k)
    return case, seqlens


def few_table_sets(seqlens):
    """Block-table sets a few-heads workload rotates through: the fewest whose
    rotation reads at least twice the L2 (so that at least the L2 passes
    between two uses of one set)."""
    kv_bytes = sum(seqlens) * 1152
    return max(1, math.ceil(2 * L2_BYTES / kv_bytes))


def torch_dtype(name):
    import torch
    return getattr(torch, name)


def oracle_rate(case, seqlens, budget_s, max_requests=None, raw=None, dequant="dequantize_kv_fp8"):
    """The float64 oracle on whole requests (all heads, every query position)
    until the time budget is used. With `raw` (the quantised rows, on any
    device) each request's rows are dequantised by the oracle first, inside the
    timed work. Returns (flops/s, description, requests done, seconds, busy
    cores)."""
    import oracle
    import synth
    s_q, causal = case.s_q, case.causal
    bt = case.block_table.numpy()
    t0, c0 = time.perf_counter(), time.process_time()
    done_flops, done = 0.0, 0
    nreq = len(seqlens) if max_requests is None else min(max_requests, len(seqlens))
    for b in range(nreq):
        rows = synth.paged_rows_index(bt[b], seqlens[b], case.page_block)
        if raw is not None:
            kv = getattr(oracle, dequant)(raw[torch_index(rows, raw.device)].cpu().numpy())
        else:
            kv = oracle.to_f64(case.kv_rows[torch_index(rows, case.kv_rows.device)].cpu())
        q = oracle.to_f64(case.q[b].cpu())
        for i in range(s_q):
            L = seqlens[b] - (s_q - 1 - i if causal else 0)
            oracle.attend(q[i], kv[:max(L, 0)], case.softmax_scale)
            done_flops += 2.0 * case.h_q * (q.shape[-1] + 512) * max(L, 0)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt, cpu = time.perf_counter() - t0, time.process_time() - c0
    what = "dequantised " if raw is not None else ""
    return (done_flops / dt, f"{done} of {len(seqlens)} requests ({what}all {case.h_q} heads, s_q={s_q})", done, dt,
            cpu / dt)


def oracle_rate_sparse(q, raw, indices, scale, budget_s, dequant="dequantize_kv_fp8"):
    """The float64 oracle on whole sparse queries: gather the query's rows by
    index, dequantise them, attend; until the time budget is used."""
    import numpy as np
    import oracle
    B, s_q = indices.shape[0], indices.shape[1]
    t0, c0 = time.perf_counter(), time.process_time()
    done_flops, done = 0.0, 0
    for n in range(B * s_q):
        b, i = n // s_q, n % s_q
        sel = indices[b, i]
        sel = sel[sel >= 0]
        kv = getattr(oracle, dequant)(raw[torch_index(sel.astype(np.int64), raw.device)].cpu().numpy())
        oracle.attend(oracle.to_f64(q[b, i].cpu()), kv, scale)
        done_flops += 2.0 * q.shape[2] * (q.shape[-1] + 512) * len(sel)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt, cpu = time.perf_counter() - t0, time.process_time() - c0
    return (done_flops / dt, f"{done} of {B * s_q} queries (index gather + dequantise + attend, all {q.shape[2]} heads)",
            done, dt, cpu / dt)


def cpu_baseline_line(rate, desc, busy):
    return {"value": round(rate / 1e12, 6), "unit": "TFLOPS", "cores": os.cpu_count(), "cores_busy": round(busy, 1),
            "kind": "oracle", "sample": f"float64 oracle on {desc} of this workload"}


def torch_index(rows, device):
    import torch
    return torch.from_numpy(rows).to(device)


def run_ours(args, w, rank, world, device):
    import torch
    import mla_latent_kv_14_gb300 as mla

    torch.cuda.set_device(device)
    case, seqlens = build_case(w, device)
    kind = w["kind"]
    s_q, causal = w["s_q"], w["causal"]
    h_q = w.get("h_q", 128)
    is_fp8 = kind in ("fp8", "sparse")
    fmt_code, row_bytes, d_k, qname, _ = FORMATS[workload_format(w)]
    q = case.q
    bt = sl = idx = None
    idx_sets = [None]
    if kind == "sparse":
        import synth
        raw = getattr(mla, qname)(case.kv_rows)              # the quantised cache, written by the library
        case.kv_rows = None
        kv = raw.view(-1, 64, 1, row_bytes)
        # the rows one step touches may fit in L2 (topk 2048: about 50 MB per
        # query position); then several seeded index sets are rotated: a
        # rotation reads at least twice the L2, and at least the L2 passes
        # between two uses of one set
        sets = [case.indices.numpy()]
        counts = [work_counts(None, s_q, False, row_bytes=row_bytes, indices=sets[0], d_k=d_k)]
        n_sets = max(1, math.ceil(2 * L2_BYTES / counts[0][2]))
        for k in range(1, n_sets):
            sets.append(synth.make_sparse_case(w["batch"], s_q, w["topk"], tokens_per_request=SPARSE_TOKENS,
                                               seed=1000 + k, with_rows=False).indices.numpy())
            counts.append(work_counts(None, s_q, False, row_bytes=row_bytes, indices=sets[-1], d_k=d_k))
        flops, algo_bytes, kv_bytes = (statistics.mean(c[j] for c in counts) for j in range(3))
        idx_sets = [torch.from_numpy(x).to(device) for x in sets]
        idx = idx_sets[0]
        meta_args = dict(batch=q.shape[0], topk=idx.shape[-1], kv_format=fmt_code, device=device)
    else:
        bt = case.block_table.to(device)
        sl = case.cache_seqlens.to(device)
        if kind == "few":
            B = len(seqlens)
            bt_sets = [bt[k * B:(k + 1) * B].contiguous() for k in range(few_table_sets(seqlens))]
            bt, sl, q = bt_sets[0], sl[:B].contiguous(), q[:B].contiguous()
        if kind == "fp8":
            raw = getattr(mla, qname)(case.kv_rows)
            kv = raw.view(case.num_blocks, 64, 1, row_bytes)
        else:
            kv = case.kvcache_paged()
        flops, algo_bytes, kv_bytes = work_counts(seqlens, s_q, causal, h_q=h_q, row_bytes=row_bytes, d_k=d_k)
        meta_args = dict(causal=causal, kv_format=fmt_code)
    out = torch.empty(q.shape[0], s_q, h_q, 512, dtype=q.dtype, device=device)
    lse = torch.empty(q.shape[0], s_q, h_q, dtype=torch.float32, device=device)
    meta, ns = mla.mla_get_metadata(sl, s_q, h_q, **meta_args)
    stream = torch.cuda.current_stream(device)
    dec_kw = dict(softmax_scale=case.softmax_scale, causal=causal, kv_format=fmt_code)

    if kind != "few":
        bt_sets = [bt]

    def step(k=0):
        m, n = mla.mla_get_metadata(sl, s_q, h_q, num_sm_parts=meta.parts, **meta_args)
        mla.mla_decode_with_kvcache(q, kv, bt_sets[k % len(bt_sets)], sl, 512, m, n, out=out, lse=lse,
                                    indices=idx_sets[k % len(idx_sets)], **dec_kw)

    # correctness gate before timing: device status must be clean
    for k in range(max(len(idx_sets), len(bt_sets))):
        step(k)
    st, bits = mla.mla_read_status(device=device)
    if st != 0:
        raise RuntimeError(f"device status {st} (bits {bits}) before timing")

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(device)
    n_sets = max(len(idx_sets), len(bt_sets))
    graph = None
    if args.graph:
        # one graph of n_sets consecutive steps (every rotated set once), with
        # the workspace fixed outside it; replayed steps/n_sets times
        ws = torch.zeros(mla.load_library().mla_workspace_size(q.shape[0], s_q, h_q, meta.parts), dtype=torch.uint8,
                         device=device)
        step_ws = step

        def step(k=0):  # noqa: F811 - the same step with a fixed workspace
            m, n = mla.mla_get_metadata(sl, s_q, h_q, num_sm_parts=meta.parts, **meta_args)
            mla.mla_decode_with_kvcache(q, kv, bt_sets[k % len(bt_sets)], sl, 512, m, n, out=out, lse=lse,
                                        indices=idx_sets[k % len(idx_sets)], workspace=ws, **dec_kw)

        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for k in range(n_sets):
                step(k)
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(n_sets):
                step(k)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(device)
        step = step_ws
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    n_timed = args.steps if graph is None else n_sets * max(1, args.steps // n_sets)
    with ClockSampler(device.index) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is None:
            for k in range(args.steps):
                step(k)
        else:
            for _ in range(n_timed // n_sets):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(device)
    elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device) * args.steps / n_timed
    if world > 1:
        torch.distributed.barrier()
    st, bits = mla.mla_read_status(device=device)
    if st != 0:
        raise RuntimeError(f"device status {st} (bits {bits}) after timing")

    # Per-kernel durations (same stream), for the roofline of the dominant
    # kernel. Every pass starts behind a spin of about 200 us on the GPU
    # (torch's sleep kernel), during which the host enqueues the pass's three
    # calls (70-80 us through the binding), so that the events bracket the
    # kernels' own execution and never a wait for the host. The inputs are the
    # timed loop's: the rows larger than L2, or rotated sets of them.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.roofline_steps)]
    for k in range(args.roofline_steps):
        torch.cuda._sleep(400_000)
        ev[k][0].record(stream)
        m, n = mla.mla_get_metadata(sl, s_q, h_q, num_sm_parts=meta.parts, **meta_args)
        ev[k][1].record(stream)
        ik, bk = idx_sets[k % len(idx_sets)], bt_sets[k % len(bt_sets)]
        mla.mla_decode_splitkv(q, kv, bk, sl, 512, m, n, out=out, lse=lse, indices=ik, **dec_kw)
        ev[k][2].record(stream)
        mla.mla_combine_splits(q, kv, bk, sl, 512, m, n, out=out, lse=lse, indices=ik, **dec_kw)
        ev[k][3].record(stream)
    torch.cuda.synchronize(device)
    t_meta = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_dec = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    t_comb = statistics.mean(e[2].elapsed_time(e[3]) for e in ev) / 1e3

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, runs the schedule and the decode, and
    # reads out/lse back into pinned host memory. Steps are pipelined the way a
    # serving loop would run them: double-buffered device inputs and outputs,
    # host->device copies on one stream, compute on another, device->host
    # copies on a third, so step k's copies overlap its neighbours' compute.
    # The time is the wall clock over all steps, synchronised on both sides.
    e2e = None
    if not args.no_e2e:
        nbuf = 2
        host_in = [q.cpu().pin_memory()] + [t.cpu().pin_memory() for t in (bt, sl, idx) if t is not None]
        host_idx = [t.cpu().pin_memory() for t in idx_sets] if idx is not None else None
        host_bt = [t.cpu().pin_memory() for t in bt_sets] if bt is not None and len(bt_sets) > 1 else None
        dev_in = [[torch.empty_like(h, device=device) for h in host_in] for _ in range(nbuf)]
        outs = [torch.empty_like(out) for _ in range(nbuf)]
        lses = [torch.empty_like(lse) for _ in range(nbuf)]
        outh = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nbuf)]
        lseh = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(nbuf)]
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        def e2e_step(k):
            j = k % nbuf
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[j])          # the compute that last read buffer j is done
                srcs = list(host_in)
                if host_idx is not None:             # the index set of this step (rotated as above)
                    srcs[-1] = host_idx[k % len(host_idx)]
                if host_bt is not None:              # the block-table set of this step
                    srcs[1] = host_bt[k % len(host_bt)]
                for hsrc, ddst in zip(srcs, dev_in[j]):
                    ddst.copy_(hsrc, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])             # out/lse buffer j has been read back
            it_ = iter(dev_in[j][1:])
            btd = next(it_) if bt is not None else None
            sld = next(it_) if sl is not None else None
            idxd = next(it_) if idx is not None else None
            m, n = mla.mla_get_metadata(sld, s_q, h_q, num_sm_parts=meta.parts, **meta_args)
            mla.mla_decode_with_kvcache(dev_in[j][0], kv, btd, sld, 512, m, n, out=outs[j], lse=lses[j],
                                        softmax_scale=case.softmax_scale, causal=causal, kv_format=fmt_code,
                                        indices=idxd)
            ev_comp[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                outh[j].copy_(outs[j], non_blocking=True)
                lseh[j].copy_(lses[j], non_blocking=True)
                ev_out[j].record(s_out)

        for k in range(max(3, args.warmup // 4)):
            e2e_step(k)
        torch.cuda.synchronize(device)
        n_e2e = max(10, args.steps // 4)
        t0 = time.perf_counter()
        for k in range(n_e2e):
            e2e_step(k)
        torch.cuda.synchronize(device)
        t_e2e = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = outh[0].numel() * outh[0].element_size() + lseh[0].numel() * 4
        e2e = {"value": round(whole_job_rate(flops, world, t_e2e) / 1e12, 3), "unit": "TFLOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(t_e2e * 1e3, 4), "pipelined_buffers": nbuf}
    return dict(elapsed=elapsed, flops=flops, algo_bytes=algo_bytes, kv_bytes=kv_bytes, t_meta=t_meta, t_dec=t_dec,
                t_comb=t_comb, clocks=clk.summary(), e2e=e2e, parts=meta.parts, case=case, seqlens=seqlens,
                raw=raw if is_fp8 else None, n_sets=max(len(idx_sets), len(bt_sets)), graph=graph is not None)


def run_absorb(args, w, world, device, hbm_peak, tc_peak, peak_src):
    """One step = mla_absorb_q + mla_up_project for T = batch*s_q tokens and
    h_q heads (d_h = 128, d_c = 512). L2 is flushed (a 512 MB write) before
    every timed step, outside the timed events, since the 32 MB of weights
    would otherwise stay in the 129 MB L2."""
    import torch
    import mla_latent_kv_14_gb300 as mla
    import synth
    T, h = w["batch"] * w["s_q"], w["h_q"]
    case = synth.make_absorb_case(T, h=h, seed=0, device=device)
    q_out = torch.zeros(T, h, 576, dtype=torch.bfloat16, device=device)
    o = torch.empty(T, h, 128, dtype=torch.bfloat16, device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flops = 2 * 2.0 * T * h * 128 * 512
    algo_bytes = 2 * (2 * h * 128 * 512 + T * h * (128 + 512 + 512 + 128))
    for _ in range(args.warmup):
        mla.mla_absorb_q(case.q_nope, case.w_uk, q_out)
        mla.mla_up_project(case.o_lat, case.w_uv, o)
    torch.cuda.synchronize(device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(device.index) as clk:
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            mla.mla_absorb_q(case.q_nope, case.w_uk, q_out)
            ev[k][1].record(stream)
            mla.mla_up_project(case.o_lat, case.w_uv, o)
            ev[k][2].record(stream)
        torch.cuda.synchronize(device)
    t_a = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_u = statistics.mean(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    t_step = max_over_ranks(t_a + t_u, world, device)
    # end to end through the public calls with host buffers (pinned), one step at a time
    hq, ho = case.q_nope.cpu().pin_memory(), case.o_lat.cpu().pin_memory()
    hq_out = torch.empty(q_out.shape, dtype=q_out.dtype).pin_memory()
    h_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    dq, do_ = torch.empty_like(case.q_nope), torch.empty_like(case.o_lat)
    n_e2e = max(10, args.steps // 4)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        dq.copy_(hq, non_blocking=True)
        do_.copy_(ho, non_blocking=True)
        mla.mla_absorb_q(dq, case.w_uk, q_out)
        mla.mla_up_project(do_, case.w_uv, o)
        hq_out.copy_(q_out, non_blocking=True)
        h_o.copy_(o, non_blocking=True)
    torch.cuda.synchronize(device)
    t_e2e = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, device)
    achieved = algo_bytes / t_step / 1e9
    bound = "hbm" if algo_bytes / (hbm_peak * 1e9) >= flops / (tc_peak * 1e12) else "tensor"
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        # the oracle's two per-head products, token by token, until the budget is used
        import oracle
        qc, ol = oracle.to_f64(case.q_nope.cpu()), oracle.to_f64(case.o_lat.cpu())
        wuk, wuv = oracle.to_f64(case.w_uk.cpu()), oracle.to_f64(case.w_uv.cpu())
        t0, c0, toks = time.perf_counter(), time.process_time(), 0
        while toks < T and time.perf_counter() - t0 < args.cpu_budget:
            oracle.absorb_q(qc[toks:toks + 1], wuk)
            oracle.up_project(ol[toks:toks + 1], wuv)
            toks += 1
        dt, busy = time.perf_counter() - t0, (time.process_time() - c0) / max(time.perf_counter() - t0, 1e-9)
        cpu = cpu_baseline_line(2 * 2.0 * toks * h * 128 * 512 / dt, f"{toks} of {T} tokens (all {h} heads)", busy)
    return {
        "metric": "absorption GEMMs (q~ = W^UK^T q^C, o = W^UV o~) throughput", "impl": "ours",
        "value": round(whole_job_rate(flops, world, t_step) / 1e12, 3), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": T, "h_q": h, "d_h": 128, "d_c": 512,
                   "parallelism": f"replicas x{world}", "l2": "flushed (512 MB write) before every timed step"},
        "kernel_us": {"absorb_q": round(t_a * 1e6, 2), "up_project": round(t_u * 1e6, 2)},
        "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "kernel": "mla_absorb_q_kernel + mla_up_project_kernel", "peak_source": f"{peak_src} hbm_gbs"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_rate(flops, world, t_e2e) / 1e12, 3), "unit": "TFLOPS",
                "h2d_bytes_per_step": int(hq.numel() * 2 + ho.numel() * 2),
                "d2h_bytes_per_step": int(hq_out.numel() * 2 + h_o.numel() * 2), "ms_per_step": round(t_e2e * 1e3, 4)},
        "clocks": clk.summary(), "gpu_launches": 2 * args.steps,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--roofline-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of a CUDA graph of the steps (schedule + decode + combine), so that the "
                         "host's per-call cost drops out of small steps")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    hbm_peak, tc_peak, tc_sus, peak_src = load_peaks()

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    device = torch.device("cuda", local)
    if world > 1:
        torch.cuda.set_device(device)
        torch.distributed.init_process_group("nccl", device_id=device)
    if w["kind"] == "absorb":
        torch.cuda.set_device(device)
        line = run_absorb(args, w, world, device, hbm_peak, tc_peak, peak_src)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    r = run_ours(args, w, rank, world, device)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    t_step = r["elapsed"] / args.steps
    tflops = whole_job_rate(r["flops"], world, t_step) / 1e12
    kv_gbs = world * r["kv_bytes"] / t_step / 1e9
    t_roof = max(r["algo_bytes"] / (hbm_peak * 1e9), r["flops"] / (tc_peak * 1e12))
    bound = "hbm" if r["algo_bytes"] / (hbm_peak * 1e9) >= r["flops"] / (tc_peak * 1e12) else "tensor"
    kname = "mla_decode_fewheads_kernel" if w["kind"] == "few" else "mla_decode_kernel"
    if bound == "hbm":
        achieved = r["algo_bytes"] / r["t_dec"] / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": stored_traffic(args.workload),
                "kernel": kname, "peak_source": f"{peak_src} hbm_gbs"}
    else:
        achieved = r["flops"] / r["t_dec"] / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(achieved / tc_peak, 4), "traffic": stored_traffic(args.workload),
                "kernel": kname, "peak_source": f"{peak_src} bf16_tflops"}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        c = r["case"]
        dq = FORMATS[workload_format(w)][4] or "dequantize_kv_fp8"
        if w["kind"] == "sparse":
            rate, desc, _, _, busy = oracle_rate_sparse(c.q, r["raw"], c.indices.numpy(), c.softmax_scale,
                                                        args.cpu_budget, dequant=dq)
        else:
            rate, desc, _, _, busy = oracle_rate(c, r["seqlens"], args.cpu_budget, raw=r["raw"], dequant=dq)
        cpu = cpu_baseline_line(rate, desc, busy)
    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp16": "fp16", "fp8_656": "fp8-e4m3 cache, fp16/bf16 MMA",
                  "fp8_528": "fp8-e4m3 cache (UE8M0 scales), bf16 MMA",
                  "fp4_288": "fp4-e2m1 cache (e4m3 scales), bf16 MMA"}[workload_format(w)],
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": w["batch"], "s_q": w["s_q"], "h_q": w.get("h_q", 128),
                   "d_qk": FORMATS[workload_format(w)][2], "d_v": 512, "page_block": 64, "causal": w["causal"],
                   "cache": {"bf16": "bf16", "fp16": "fp16", "fp8_656": "fp8-656B", "fp8_528": "fp8-528B",
                             "fp4_288": "fp4-288B"}[workload_format(w)],
                   "seqlens": (f"topk {w['topk']} of {SPARSE_TOKENS} per request, 5% -1" if w["kind"] == "sparse"
                               else f"all {w['lens'][1]}" if w["lens"][0] == "fixed"
                               else f"uniform [{w['lens'][1]},{w['lens'][2]}] seed 2"),
                   "parallelism": f"replicas x{world}", "num_sm_parts": r["parts"],
                   "launch": "CUDA graph replays" if r["graph"] else "calls on the stream",
                   "l2": ("inputs larger than L2 (KV cache %.0f MB per replica)" % (r["kv_bytes"] / 1e6)
                          if r["n_sets"] == 1 else
                          "inputs larger than L2: %d %s sets rotated, %.0f MB of rows each"
                          % (r["n_sets"], "index" if w["kind"] == "sparse" else "block-table", r["kv_bytes"] / 1e6))},
        "kv_gbs": round(kv_gbs, 1), "algo_gbs": round(world * r["algo_bytes"] / t_step / 1e9, 1),
        "roofline_time_frac": round(t_roof / t_step, 4),
        "kernel_us": {"metadata": round(r["t_meta"] * 1e6, 2), "decode": round(r["t_dec"] * 1e6, 2),
                      "combine": round(r["t_comb"] * 1e6, 2)},
        "roofline": roof, "cpu_baseline": cpu, "e2e": r["e2e"], "clocks": r["clocks"],
        "gpu_launches": 3 * args.steps,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, w, rank, world):
    """The oracle (float64, host cores) on bounded samples of the workload."""
    if world > 1 and rank != 0:
        return
    import numpy as np
    import oracle
    import synth
    budget = 120.0 / (args.steps + args.warmup)     # keep the whole run within ~2 minutes
    metric = METRIC
    if w["kind"] == "absorb":
        # the oracle's two per-head products on a bounded number of tokens
        T, h = w["batch"] * w["s_q"], w["h_q"]
        ab = synth.make_absorb_case(T, h=h, seed=0)
        qc, ol = oracle.to_f64(ab.q_nope), oracle.to_f64(ab.o_lat)
        wuk, wuv = oracle.to_f64(ab.w_uk), oracle.to_f64(ab.w_uv)
        t0 = time.perf_counter()
        oracle.absorb_q(qc[:1], wuk)
        oracle.up_project(ol[:1], wuv)
        toks = int(max(1, min(T, budget / max(time.perf_counter() - t0, 1e-6))))
        run = lambda: (oracle.absorb_q(qc[:toks], wuk), oracle.up_project(ol[:toks], wuv))
        flops = 2 * 2.0 * toks * h * 128 * 512
        sample = f"float64 oracle, {toks} of {T} tokens x {h} heads per step"
        metric = "absorption GEMMs (q~ = W^UK^T q^C, o = W^UV o~) throughput"
    else:
        d_k = FORMATS[workload_format(w)][2]
        if w["kind"] == "sparse":
            # one query of one request: its top-k rows gathered
            sp = synth.make_sparse_case(1, 1, w["topk"], tokens_per_request=SPARSE_TOKENS, seed=0, d_k=d_k)
            sel = sp.indices.numpy()[0, 0]
            kv = oracle.to_f64(sp.kv_rows)[sel[sel >= 0]]
            q = oracle.to_f64(sp.q[0])
            scale = sp.softmax_scale
        else:
            seqlens = workload_seqlens(w)
            case = synth.make_dense_case(seqlens[:1], s_q=w["s_q"], h_q=w.get("h_q", 128), causal=w["causal"],
                                         seed=0, d_k=d_k)
            rows = synth.paged_rows_index(case.block_table.numpy()[0], seqlens[0], 64)
            kv = oracle.to_f64(case.kv_rows)[rows]
            q = oracle.to_f64(case.q[0])
            scale = case.softmax_scale
        L, hq = kv.shape[0], q.shape[1]
        t0 = time.perf_counter()
        oracle.attend(q[0], kv, scale)
        t_full = time.perf_counter() - t0
        heads = int(max(1, min(hq, hq * budget / max(t_full, 1e-6))))
        run = lambda: oracle.attend(q[0, :heads], kv, scale)
        flops = 2.0 * heads * (d_k + 512) * L
        sample = f"float64 oracle, one request of {L} tokens x {heads} heads per step (s_q position 0)"
    for _ in range(args.warmup):
        run()
    t0, c0 = time.perf_counter(), time.process_time()
    for _ in range(args.steps):
        run()
    busy = (time.process_time() - c0) / max(time.perf_counter() - t0, 1e-9)
    dt = (time.perf_counter() - t0) / args.steps
    val = flops / dt / 1e12
    line = {"impl": "reference", "metric": metric, "value": round(val, 6), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": w["batch"], "s_q": w["s_q"], "h_q": w.get("h_q", 128)},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOPS", "cores": os.cpu_count(),
                             "cores_busy": round(busy, 1), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
