"""GPU parity of the per-head GEMMs around the decode kernel against the
float64 oracle: q~ = W^UK_i^T q^C (mla_absorb_q) and o = W^UV_i o~
(mla_up_project), "矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA" §六 '吸收'.

Outputs are rounded once to the 16-bit input type, so the bar is the one the
attention tests use: |d| <= 8e-3 + 1e-2 |ref| for values of order one. The
last test chains absorb -> decode -> up-project and compares with naive
per-head attention over the un-absorbed keys and values.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_14_gb300")
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.load_library()


def _close(got, ref, what):
    got = got.double().cpu().numpy()
    err = np.abs(got - ref)
    bad = err > 8e-3 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside the bar, max err {err.max():.3g}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("tokens,h", [(1, 128), (64, 128), (200, 16), (130, 3)])
def test_absorb_q(tokens, h, dtype):
    case = synth.make_absorb_case(tokens, h=h, dtype=dtype, seed=tokens + h)
    q_out = torch.full((tokens, h, 576), 7.0, dtype=dtype, device=DEV)   # RoPE dims must survive
    mla.mla_absorb_q(case.q_nope.to(DEV), case.w_uk.to(DEV), q_out)
    torch.cuda.synchronize()
    ref = oracle.absorb_q(oracle.to_f64(case.q_nope), oracle.to_f64(case.w_uk))
    _close(q_out[..., :512], ref, f"absorb T={tokens} h={h} {dtype}")
    assert (q_out[..., 512:].float() == 7.0).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("tokens,h", [(1, 128), (64, 128), (200, 16), (130, 3)])
def test_up_project(tokens, h, dtype):
    case = synth.make_absorb_case(tokens, h=h, dtype=dtype, seed=100 + tokens + h)
    o = mla.mla_up_project(case.o_lat.to(DEV), case.w_uv.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.up_project(oracle.to_f64(case.o_lat), oracle.to_f64(case.w_uv))
    _close(o, ref, f"up-project T={tokens} h={h} {dtype}")


def test_empty_and_bad_args():
    case = synth.make_absorb_case(1, h=2)
    q_out = torch.zeros(0, 2, 576, dtype=torch.bfloat16, device=DEV)
    mla.mla_absorb_q(case.q_nope[:0].to(DEV), case.w_uk.to(DEV), q_out)   # tokens = 0: nothing to do
    lib = mla.load_library()
    w = case.w_uk.to(DEV)
    assert lib.mla_absorb_q(w.data_ptr(), w.data_ptr(), w.data_ptr(), -1, 2, 0, None, None) == 1
    assert lib.mla_up_project(w.data_ptr(), w.data_ptr(), w.data_ptr(), 4, 2, 5, None, None) == 1
    assert lib.mla_up_project(w.data_ptr() + 2, w.data_ptr(), w.data_ptr(), 4, 2, 0, None, None) == 1


def test_absorbed_chain_equals_naive_per_head_attention():
    """absorb -> decode -> up-project on the GPU against naive per-head attention
    with k_i = [W^UK_i c; k^R] and v_i = W^UV_i c, in float64 from the same
    16-bit inputs."""
    B, h, L = 2, 128, 200
    dense = synth.make_dense_case([L, 77], h_q=h, seed=5)
    ab = synth.make_absorb_case(B, h=h, seed=6)
    q_rope = dense.q[:, 0, :, 512:]                                  # [B, h, 64]
    q = torch.empty(B, 1, h, 576, dtype=torch.bfloat16, device=DEV)
    q[:, 0, :, 512:] = q_rope.to(DEV)
    mla.mla_absorb_q(ab.q_nope.to(DEV), ab.w_uk.to(DEV), q.view(B, h, 576))
    sl = dense.cache_seqlens.to(DEV)
    meta, ns = mla.mla_get_metadata(sl, 1, h)
    o_lat, lse = mla.mla_decode_with_kvcache(q, dense.kvcache_paged().to(DEV), dense.block_table.to(DEV), sl, 512,
                                             meta, ns, softmax_scale=dense.softmax_scale)
    o = mla.mla_up_project(o_lat.view(B, h, 512), ab.w_uv.to(DEV))
    torch.cuda.synchronize()
    rows = oracle.to_f64(dense.kv_rows)
    wuk, wuv = oracle.to_f64(ab.w_uk), oracle.to_f64(ab.w_uv)
    qc, qr = oracle.to_f64(ab.q_nope), oracle.to_f64(q_rope)
    bt = dense.block_table.numpy()
    for b, Lb in enumerate(dense.cache_seqlens.numpy()):
        kv = rows[synth.paged_rows_index(bt[b], int(Lb), 64)]
        c, kr = kv[:, :512], kv[:, 512:]
        ref = np.empty((h, 128))
        for i in range(h):
            k_i = np.concatenate([c @ wuk[i].T, kr], axis=1)            # [L, 128 + 64]
            s = dense.softmax_scale * (k_i @ np.concatenate([qc[b, i], qr[b, i]]))
            p = np.exp(s - s.max())
            ref[i] = (p @ (c @ wuv[i].T)) / p.sum()
        _close(o[b], ref, f"absorbed chain b={b}")
