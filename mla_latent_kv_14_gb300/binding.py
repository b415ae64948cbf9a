"""ctypes binding of libmla (include/mla.h). Marshalling only: every step of the
decode runs in the library's CUDA kernels; PyTorch supplies device memory and
streams. Nothing here computes attention, and there is no fallback path: if
the shared library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "stale metadata",
                4: "out-of-range page or index skipped", 5: "device wait timed out", 6: "CUDA error",
                7: "FP8 path: a value beyond fp16 range was saturated"}
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1}

_lib = None
_lib_lock = threading.Lock()


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} (status {status})")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmla.so (built by ``mla_latent_kv_14_gb300.build``)."""
    global _lib
    with _lib_lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libmla.so not built at {p}: run `python -m mla_latent_kv_14_gb300.build`")
        lib = ctypes.CDLL(p)
        c = ctypes
        vp, i32p = c.c_void_p, c.c_void_p
        lib.mla_status_string.restype = c.c_char_p
        lib.mla_status_string.argtypes = [c.c_int]
        lib.mla_num_sm_parts.restype = c.c_int
        lib.mla_num_sm_parts.argtypes = [c.c_int]
        lib.mla_num_sm_parts_for.restype = c.c_int
        lib.mla_num_sm_parts_for.argtypes = [c.c_int, c.c_int]
        lib.mla_metadata_size.restype = c.c_size_t
        lib.mla_metadata_size.argtypes = [c.c_int, c.c_int, c.c_int]
        lib.mla_workspace_size.restype = c.c_size_t
        lib.mla_workspace_size.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int]
        lib.mla_get_metadata.restype = c.c_int
        lib.mla_get_metadata.argtypes = [i32p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                         c.c_int, c.c_int, vp, i32p, vp]
        lib.mla_decode_with_kvcache.restype = c.c_int
        lib.mla_decode_with_kvcache.argtypes = [vp, c.c_int, vp, c.c_int64, c.c_int, i32p, c.c_int, i32p, c.c_int,
                                                c.c_int, c.c_int, c.c_int, vp, i32p, c.c_int, c.c_float, c.c_int,
                                                c.c_int, i32p, c.c_int, vp, vp, vp, c.c_size_t, vp]
        for name in ("mla_decode_splitkv", "mla_combine_splits"):
            f = getattr(lib, name)
            f.restype = c.c_int
            f.argtypes = lib.mla_decode_with_kvcache.argtypes
        lib.mla_decode_with_kvcache_noalloc.restype = c.c_int
        lib.mla_decode_with_kvcache_noalloc.argtypes = lib.mla_decode_with_kvcache.argtypes[:-3] + [vp, vp]
        for name in ("mla_quantize_kv_fp8", "mla_quantize_kv_fp8_528", "mla_quantize_kv_fp4_288"):
            f = getattr(lib, name)
            f.restype = c.c_int
            f.argtypes = [vp, vp, c.c_int64, vp]
        lib.mla_read_status.restype = c.c_int
        lib.mla_read_status.argtypes = [vp, vp, c.POINTER(c.c_uint32)]
        for name in ("mla_absorb_q", "mla_up_project"):
            f = getattr(lib, name)
            f.restype = c.c_int
            f.argtypes = [vp, vp, vp, c.c_int, c.c_int, c.c_int, vp, vp]
        lib.mla_set_test_stall.restype = None
        lib.mla_set_test_stall.argtypes = [c.c_uint32]
        if path is None:
            _lib = lib
        return lib


def _dev(device=None) -> torch.device:
    """A cuda device with an explicit index (the current one if unspecified)."""
    d = torch.device("cuda") if device is None else torch.device(device)
    if d.index is None:
        d = torch.device("cuda", torch.cuda.current_device())
    return d


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MLAError(status, where)


def mla_num_sm_parts(device=None, h_q: int = 128) -> int:
    """Default number of SM parts of the decode kernel for `h_q` query heads."""
    n = load_library().mla_num_sm_parts_for(_dev(device).index, h_q)
    if n <= 0:
        raise MLAError(2 if n < 0 else 6, "mla_num_sm_parts")
    return n


class Metadata:
    """Split-KV schedule from :func:`mla_get_metadata` (device tensors)."""

    def __init__(self, meta: torch.Tensor, num_splits: torch.Tensor, parts: int, key: tuple):
        self.meta = meta
        self.num_splits = num_splits
        self.parts = parts
        self.key = key


# cache row formats (the kv_format argument; is_fp8=True is KV_FP8_656)
KV_16BIT, KV_FP8_656, KV_FP8_528, KV_FP4_288 = 0, 1, 2, 3
ROW_WIDTH = {KV_16BIT: 576, KV_FP8_656: 576, KV_FP8_528: 512, KV_FP4_288: 512}   # query / key width


def _kv_format(is_fp8: bool, kv_format: Optional[int]) -> int:
    if kv_format is None:
        return KV_FP8_656 if is_fp8 else KV_16BIT
    if kv_format not in ROW_WIDTH:
        raise MLAError(1, f"unknown kv_format {kv_format}")
    return int(kv_format)


def mla_get_metadata(cache_seqlens: Optional[torch.Tensor], s_q: int, h_q: int = 128, *, batch: Optional[int] = None,
                     topk: int = 0, is_fp8: bool = False, causal: bool = False, page_block: int = 64,
                     num_sm_parts: Optional[int] = None, device=None,
                     kv_format: Optional[int] = None) -> Tuple[Metadata, torch.Tensor]:
    """Compute the split-KV schedule on the device (no host sync)."""
    lib = load_library()
    fmt = _kv_format(is_fp8, kv_format)
    if cache_seqlens is not None:
        batch = int(cache_seqlens.shape[0])
        device = cache_seqlens.device
        assert cache_seqlens.dtype == torch.int32 and cache_seqlens.is_contiguous()
    assert batch is not None and device is not None
    device = _dev(device)
    parts = num_sm_parts or mla_num_sm_parts(device, h_q)
    nbytes = lib.mla_metadata_size(batch, s_q, parts)
    meta = torch.empty((nbytes + 3) // 4, dtype=torch.int32, device=device)
    num_splits = torch.empty(batch * s_q + 1, dtype=torch.int32, device=device)
    st = lib.mla_get_metadata(_ptr(cache_seqlens), batch, s_q, h_q, 1, topk, fmt, int(causal), page_block,
                              parts, _ptr(meta), _ptr(num_splits), _stream(device))
    _check(st, "mla_get_metadata")
    return Metadata(meta, num_splits, parts, (batch, s_q, h_q, topk, fmt, bool(causal))), num_splits


_ws_cache = {}
_ws_lock = threading.Lock()


def workspace_for(device: torch.device, nbytes: int) -> torch.Tensor:
    """A zero-initialised workspace cached per (device, stream); grown on demand."""
    device = _dev(device)
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def mla_decode_with_kvcache(q: torch.Tensor, kvcache: torch.Tensor, block_table: Optional[torch.Tensor],
                            cache_seqlens: Optional[torch.Tensor], head_dim_v: int, metadata: Metadata,
                            num_splits: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                            causal: bool = False, is_fp8: bool = False, indices: Optional[torch.Tensor] = None,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, kv_format: Optional[int] = None,
                            _entry: str = "mla_decode_with_kvcache") -> Tuple[torch.Tensor, torch.Tensor]:
    """out [B, s_q, h_q, 512] (q dtype), lse [B, s_q, h_q] fp32 (natural log).
    ``kv_format`` picks the cache row format (KV_*); q is [B, s_q, h_q, 576],
    or 512 wide with the V4.1 rows (KV_FP8_528, KV_FP4_288)."""
    lib = load_library()
    fmt = _kv_format(is_fp8, kv_format)
    B, s_q, h_q, d_k = q.shape
    assert d_k == ROW_WIDTH[fmt] and q.is_contiguous() and kvcache.is_contiguous()
    dev = _dev(q.device)
    num_blocks, page_block = int(kvcache.shape[0]), int(kvcache.shape[1])
    if softmax_scale is None:
        softmax_scale = d_k ** -0.5
    if num_splits is None:
        num_splits = metadata.num_splits
    topk = int(indices.shape[-1]) if indices is not None else 0
    if out is None:
        out = torch.empty(B, s_q, h_q, head_dim_v, dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=dev)
    wsb = lib.mla_workspace_size(B, s_q, h_q, metadata.parts)
    if workspace is None:
        workspace = workspace_for(dev, wsb)
    max_blocks = int(block_table.shape[1]) if block_table is not None else 0
    st = getattr(lib, _entry)(
        _ptr(q), DTYPE_CODES[q.dtype], _ptr(kvcache), num_blocks, page_block, _ptr(block_table), max_blocks,
        _ptr(cache_seqlens), B, s_q, h_q, head_dim_v, _ptr(metadata.meta), _ptr(num_splits), metadata.parts,
        float(softmax_scale), int(causal), fmt, _ptr(indices), topk, _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel(), _stream(dev))
    _check(st, _entry)
    return out, lse


def mla_decode_splitkv(*args, **kw):
    """Only the split-KV kernel of :func:`mla_decode_with_kvcache`."""
    return mla_decode_with_kvcache(*args, _entry="mla_decode_splitkv", **kw)


def mla_combine_splits(*args, **kw):
    """Only the combine of :func:`mla_decode_with_kvcache` (after mla_decode_splitkv)."""
    return mla_decode_with_kvcache(*args, _entry="mla_combine_splits", **kw)


def mla_decode_with_kvcache_noalloc(q: torch.Tensor, kvcache: torch.Tensor, block_table: Optional[torch.Tensor],
                                    cache_seqlens: Optional[torch.Tensor], head_dim_v: int, metadata: Metadata,
                                    num_splits: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                                    causal: bool = False, is_fp8: bool = False,
                                    indices: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                                    lse: Optional[torch.Tensor] = None,
                                    status: Optional[torch.Tensor] = None,
                                    kv_format: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Decode using the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory on demand). ``out``/``lse``
    /``status`` are allocated here only when not given."""
    lib = load_library()
    fmt = _kv_format(is_fp8, kv_format)
    B, s_q, h_q, d_k = q.shape
    assert d_k == ROW_WIDTH[fmt] and q.is_contiguous() and kvcache.is_contiguous()
    dev = _dev(q.device)
    num_blocks, page_block = int(kvcache.shape[0]), int(kvcache.shape[1])
    if softmax_scale is None:
        softmax_scale = d_k ** -0.5
    if num_splits is None:
        num_splits = metadata.num_splits
    topk = int(indices.shape[-1]) if indices is not None else 0
    if out is None:
        out = torch.empty(B, s_q, h_q, head_dim_v, dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=dev)
    max_blocks = int(block_table.shape[1]) if block_table is not None else 0
    st = lib.mla_decode_with_kvcache_noalloc(
        _ptr(q), DTYPE_CODES[q.dtype], _ptr(kvcache), num_blocks, page_block, _ptr(block_table), max_blocks,
        _ptr(cache_seqlens), B, s_q, h_q, head_dim_v, _ptr(metadata.meta), _ptr(num_splits), metadata.parts,
        float(softmax_scale), int(causal), fmt, _ptr(indices), topk, _ptr(out), _ptr(lse), _ptr(status),
        _stream(dev))
    _check(st, "mla_decode_with_kvcache_noalloc")
    return out, lse


def mla_quantize_kv_fp8(kv: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 rows [..., 576] -> uint8 rows [..., 656] (the FP8 cache layout)."""
    lib = load_library()
    assert kv.dtype == torch.bfloat16 and kv.shape[-1] == 576 and kv.is_contiguous()
    n = kv.numel() // 576
    if out is None:
        out = torch.empty(*kv.shape[:-1], 656, dtype=torch.uint8, device=kv.device)
    st = lib.mla_quantize_kv_fp8(_ptr(kv), _ptr(out), n, _stream(kv.device))
    _check(st, "mla_quantize_kv_fp8")
    return out


def _quantize_v41(name: str, row_bytes: int, kv: torch.Tensor, out: Optional[torch.Tensor]) -> torch.Tensor:
    lib = load_library()
    assert kv.dtype == torch.bfloat16 and kv.shape[-1] == 512 and kv.is_contiguous()
    n = kv.numel() // 512
    if out is None:
        out = torch.empty(*kv.shape[:-1], row_bytes, dtype=torch.uint8, device=kv.device)
    st = getattr(lib, name)(_ptr(kv), _ptr(out), n, _stream(kv.device))
    _check(st, name)
    return out


def mla_quantize_kv_fp8_528(kv: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 rows [..., 512] -> uint8 rows [..., 528] (V4.1: e4m3 + UE8M0 per 32)."""
    return _quantize_v41("mla_quantize_kv_fp8_528", 528, kv, out)


def mla_quantize_kv_fp4_288(kv: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """bf16 rows [..., 512] -> uint8 rows [..., 288] (e2m1 + e4m3 per 16)."""
    return _quantize_v41("mla_quantize_kv_fp4_288", 288, kv, out)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return 0
    if t.dtype == torch.float16:
        return 1
    raise MLAError(1, f"unsupported dtype {t.dtype}")


def mla_absorb_q(q_nope: torch.Tensor, w_uk: torch.Tensor, q_out: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """q~ = W^UK_i^T q^C per head: q_nope [..., h, 128], w_uk [h, 128, 512] ->
    dims [0, 512) of q_out [..., h, 576] (allocated if not given; its RoPE dims
    are the caller's). ``status``: optional device status word (read it with
    :func:`mla_read_status`)."""
    lib = load_library()
    h = q_nope.shape[-2]
    assert q_nope.shape[-1] == 128 and tuple(w_uk.shape) == (h, 128, 512)
    assert q_nope.is_contiguous() and w_uk.is_contiguous() and w_uk.dtype == q_nope.dtype
    tokens = q_nope.numel() // (h * 128)
    if q_out is None:
        q_out = torch.zeros(*q_nope.shape[:-1], 576, dtype=q_nope.dtype, device=q_nope.device)
    assert q_out.is_contiguous() and q_out.dtype == q_nope.dtype and q_out.numel() == tokens * h * 576
    st = lib.mla_absorb_q(_ptr(q_nope), _ptr(w_uk), _ptr(q_out), tokens, h, _dtype_code(q_nope), _ptr(status),
                          _stream(q_nope.device))
    _check(st, "mla_absorb_q")
    return q_out


def mla_up_project(o_lat: torch.Tensor, w_uv: torch.Tensor, o_out: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """o = W^UV_i o~ per head: o_lat [..., h, 512], w_uv [h, 128, 512] -> [..., h, 128].
    ``status``: optional device status word (read it with :func:`mla_read_status`)."""
    lib = load_library()
    h = o_lat.shape[-2]
    assert o_lat.shape[-1] == 512 and tuple(w_uv.shape) == (h, 128, 512)
    assert o_lat.is_contiguous() and w_uv.is_contiguous() and w_uv.dtype == o_lat.dtype
    tokens = o_lat.numel() // (h * 512)
    if o_out is None:
        o_out = torch.empty(*o_lat.shape[:-1], 128, dtype=o_lat.dtype, device=o_lat.device)
    assert o_out.is_contiguous() and o_out.dtype == o_lat.dtype and o_out.numel() == tokens * h * 128
    st = lib.mla_up_project(_ptr(o_lat), _ptr(w_uv), _ptr(o_out), tokens, h, _dtype_code(o_lat), _ptr(status),
                            _stream(o_lat.device))
    _check(st, "mla_up_project")
    return o_out


def mla_read_status(workspace: Optional[torch.Tensor] = None, device=None) -> Tuple[int, int]:
    """Synchronise and return (status, bits) of a workspace, clearing it."""
    lib = load_library()
    dev = _dev(device)
    if workspace is None:
        workspace = workspace_for(dev, 256)
    bits = ctypes.c_uint32(0)
    st = lib.mla_read_status(_ptr(workspace), _stream(dev), ctypes.byref(bits))
    return st, int(bits.value)


def mla_set_test_stall(cycles: int) -> None:
    """Test hook of the time-out path: while non-zero, every decode and
    absorption launch first waits ``cycles`` SM cycles on a barrier nothing
    arrives at, records a wait time-out and skips its work. 0 turns it off."""
    load_library().mla_set_test_stall(int(cycles))
