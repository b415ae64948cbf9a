"""CPU checks of the C ABI: the library loads without a GPU, exports every
entry point include/mla.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    import mla_latent_kv_14_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from mla_latent_kv_14_gb300 import build
        build.build()
    return m.load_library()


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["mla_get_metadata", "mla_decode_with_kvcache", "mla_decode_splitkv", "mla_combine_splits", "mla_quantize_kv_fp8", "mla_read_status",
                 "mla_absorb_q", "mla_up_project", "mla_decode_with_kvcache_noalloc",
                 "mla_metadata_size", "mla_workspace_size", "mla_num_sm_parts", "mla_status_string",
                 "mla_set_test_stall", "mla_quantize_kv_fp8_528", "mla_quantize_kv_fp4_288"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    import mla_latent_kv_14_gb300 as m
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mla_\w+)", out))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    for n in declared_symbols():
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(8):
        assert lib.mla_status_string(code)
        assert b"unknown" not in lib.mla_status_string(code)
    assert b"unknown" in lib.mla_status_string(99)


def test_sizes(lib):
    assert lib.mla_metadata_size(64, 1, 76) == 4 * (16 + 8 * 76)
    ws = lib.mla_workspace_size(64, 1, 128, 76)
    assert ws == 256 + (64 + 76) * 128 * 512 * 4 + (64 + 76) * 128 * 4 + 64 * 16
    assert lib.mla_workspace_size(0, 1, 128, 76) == 0


FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: checks fail first


def _decode(lib, **kw):
    a = dict(q=FAKE, q_dtype=0, kv=FAKE, num_blocks=8, page_block=64, bt=FAKE, max_blocks=8, sl=FAKE, batch=2,
             s_q=1, h_q=128, dv=512, meta=FAKE, ns=FAKE, parts=4, scale=576 ** -0.5, causal=0, fp8=0, idx=None,
             topk=0, out=FAKE, lse=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.mla_decode_with_kvcache(a["q"], a["q_dtype"], a["kv"], a["num_blocks"], a["page_block"], a["bt"],
                                       a["max_blocks"], a["sl"], a["batch"], a["s_q"], a["h_q"], a["dv"], a["meta"],
                                       a["ns"], a["parts"], a["scale"], a["causal"], a["fp8"], a["idx"], a["topk"],
                                       a["out"], a["lse"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dv=256), 1),                                  # head_dim_v must be 512
    (dict(page_block=32), 1),
    (dict(q=None), 1),
    (dict(q_dtype=7), 1),
    (dict(idx=FAKE, topk=2048, causal=1), 1),           # causal with indices
    (dict(idx=FAKE, topk=0), 1),                        # indices without topk
    (dict(bt=None), 1),                                 # dense needs a block table
    (dict(q=ctypes.c_void_p((1 << 20) + 2)), 1),        # misaligned q
    (dict(ws=ctypes.c_void_p((1 << 20) + 16)), 1),      # workspace needs 256-B alignment
    (dict(wsb=100), 1),                                 # workspace too small
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(batch=0), 1),
    (dict(h_q=64), 2),                                  # not implemented
    (dict(fp8=4), 1),                                   # no such cache format
    (dict(fp8=-1), 1),
    (dict(fp8=2, q_dtype=1), 2),                        # quantised rows pair with bf16 queries
    (dict(fp8=3, q_dtype=1), 2),
    (dict(idx=FAKE, topk=64, fp8=0), 2),                # token-sparse decode reads quantised rows
])
def test_decode_argument_checks(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_metadata_argument_checks(lib):
    f = lib.mla_get_metadata
    assert f(FAKE, 2, 1, 128, 2, 0, 0, 0, 64, 4, FAKE, FAKE, None) == 1        # h_kv != 1
    assert f(FAKE, 2, 1, 128, 1, 0, 0, 0, 32, 4, FAKE, FAKE, None) == 1        # page_block
    assert f(None, 2, 1, 128, 1, 0, 0, 0, 64, 4, FAKE, FAKE, None) == 1        # dense needs lengths
    assert f(None, 2, 1, 128, 1, 64, 1, 1, 64, 4, FAKE, FAKE, None) == 1       # sparse + causal
    assert f(FAKE, 2, 1, 128, 1, 0, 0, 0, 64, 0, FAKE, FAKE, None) == 1        # parts
    assert f(FAKE, 2, 1, 128, 1, 0, 4, 0, 64, 4, FAKE, FAKE, None) == 1        # no such cache format
    assert f(FAKE, 2, 1, 16, 1, 0, 2, 0, 64, 4, FAKE, FAKE, None) == 2         # few heads: 16-bit caches


@pytest.mark.parametrize("name", ["mla_quantize_kv_fp8", "mla_quantize_kv_fp8_528", "mla_quantize_kv_fp4_288"])
def test_quantize_argument_checks(lib, name):
    f = getattr(lib, name)
    assert f(FAKE, FAKE, -1, None) == 1
    assert f(ctypes.c_void_p((1 << 20) + 8), FAKE, 4, None) == 1
    assert f(FAKE, ctypes.c_void_p((1 << 20) + 8), 4, None) == 1
    assert f(None, FAKE, 4, None) == 1
    assert f(FAKE, FAKE, 0, None) == 0


@pytest.mark.parametrize("name", ["mla_absorb_q", "mla_up_project"])
def test_absorption_argument_checks(lib, name):
    """Bad sizes, dtypes, null or misaligned pointers are rejected before any
    device call; tokens = 0 is a no-op."""
    f = getattr(lib, name)
    mis = ctypes.c_void_p((1 << 20) + 8)
    assert f(FAKE, FAKE, FAKE, -1, 128, 0, None, None) == 1          # negative token count
    assert f(FAKE, FAKE, FAKE, 4, 0, 0, None, None) == 1             # no heads
    assert f(FAKE, FAKE, FAKE, 4, 128, 7, None, None) == 1           # unknown dtype
    assert f(None, FAKE, FAKE, 4, 128, 0, None, None) == 1           # null input
    assert f(FAKE, None, FAKE, 4, 128, 0, None, None) == 1           # null weights
    assert f(FAKE, FAKE, None, 4, 128, 0, None, None) == 1           # null output
    assert f(mis, FAKE, FAKE, 4, 128, 0, None, None) == 1            # misaligned input
    assert f(FAKE, mis, FAKE, 4, 128, 1, None, None) == 1            # misaligned weights
    assert f(FAKE, FAKE, mis, 4, 128, 0, None, None) == 1            # misaligned output
    assert f(FAKE, FAKE, FAKE, 4, 128, 0, ctypes.c_void_p((1 << 20) + 2), None) == 1  # misaligned status word
    assert f(None, None, None, 0, 128, 0, None, None) == 0           # nothing to do


def _noalloc(lib, **kw):
    a = dict(q=FAKE, q_dtype=0, kv=FAKE, num_blocks=8, page_block=64, bt=FAKE, max_blocks=8, sl=FAKE, batch=2,
             s_q=1, h_q=128, dv=512, meta=FAKE, ns=FAKE, parts=4, scale=576 ** -0.5, causal=0, fp8=0, idx=None,
             topk=0, out=FAKE, lse=FAKE, status=None, stream=None)
    a.update(kw)
    return lib.mla_decode_with_kvcache_noalloc(
        a["q"], a["q_dtype"], a["kv"], a["num_blocks"], a["page_block"], a["bt"], a["max_blocks"], a["sl"],
        a["batch"], a["s_q"], a["h_q"], a["dv"], a["meta"], a["ns"], a["parts"], a["scale"], a["causal"], a["fp8"],
        a["idx"], a["topk"], a["out"], a["lse"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dv=256), 1),
    (dict(q=None), 1),
    (dict(idx=FAKE, topk=2048, causal=1), 1),
    (dict(bt=None), 1),
    (dict(q=ctypes.c_void_p((1 << 20) + 2)), 1),
    (dict(status=ctypes.c_void_p((1 << 20) + 2)), 1),   # misaligned status word
    (dict(batch=4096, parts=76), 1),                    # scratch beyond the fixed array
    (dict(h_q=64), 2),
])
def test_noalloc_rejects_before_any_device_call(lib, kw, code):
    """Every argument check of the allocation-free entry point runs before it
    touches the device: on a host without a GPU any CUDA call would fail with
    MLA_ERR_CUDA (6), so the argument error must come back instead."""
    assert _noalloc(lib, **kw) == code


def test_set_test_stall_is_host_only(lib):
    lib.mla_set_test_stall(1000)
    lib.mla_set_test_stall(0)
