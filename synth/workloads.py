"""Seeded generators for the decode workloads.

Shapes follow the MLA decode call described in "FlashMLA 实战：MLA 注意力加速指南"
(§最小调用) and "矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA" (§六 'cache 账本',
§八 sparse indices): a query of h_q heads x 576 (512 absorbed latent + 64 RoPE),
one shared 576-wide latent row per cached token, a paged cache of
``page_block``-token pages addressed through a block table, and for the sparse
mode an index list with -1 padding.

Seeds: 0 -> q and cache values, 1 -> block-table permutation, 2 -> sequence
lengths, 3 -> sparse indices, 4 -> outlier channels. Everything is produced on
the CPU with torch's seeded generator (bf16/fp16 rounding is torch's) unless a
``device`` is given, in which case the large tensors are drawn on that device
with a device generator (different stream, same distribution).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

D_K = 576          # latent (512) + decoupled RoPE (64)
D_V = 512          # value = the latent part of the row
D_ROPE = 64
FP8_ROW_BYTES = 656  # 512 e4m3 + 4 fp32 scales + 64 bf16


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def uniform_seqlens(batch: int, lo: int, hi: int, seed: int = 2) -> np.ndarray:
    """Sequence lengths drawn uniformly from the integers in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def make_latent_rows(n_rows: int, dtype=torch.bfloat16, seed: int = 0,
                     outlier_channels: int = 0, outlier_gain: float = 8.0,
                     device="cpu", d_k: int = D_K) -> torch.Tensor:
    """``n_rows`` x ``d_k`` cache rows ~ N(0,1) in ``dtype`` (576, or 512 for
    the V4.1 rows whose 512 values hold latent and RoPE together).

    With ``outlier_channels`` > 0, that many seeded latent channels of every
    row (distinct, in [0, 512)) are multiplied by ``outlier_gain`` before the
    rounding to ``dtype``.
    """
    g = _gen(seed, device)
    x = torch.randn(n_rows, d_k, generator=g, device=device, dtype=torch.float32)
    if outlier_channels > 0:
        go = _gen(seed + 4, device)
        # per-row distinct channels: top-k of a random key per (row, channel)
        keys = torch.rand(n_rows, D_V, generator=go, device=device)
        ch = keys.topk(outlier_channels, dim=1).indices
        x[:, :D_V].scatter_(1, ch, x[:, :D_V].gather(1, ch) * outlier_gain)
    return x.to(dtype)


def paged_rows_index(block_table: np.ndarray, seqlen: int, page_block: int) -> np.ndarray:
    """Absolute cache-row index of tokens 0..seqlen-1 of one request."""
    t = np.arange(seqlen)
    return block_table[t // page_block].astype(np.int64) * page_block + t % page_block


@dataclasses.dataclass
class DenseCase:
    q: torch.Tensor              # [B, s_q, h_q, 576]
    kv_rows: torch.Tensor        # [num_blocks * page_block, 576] (bf16/fp16)
    block_table: torch.Tensor    # [B, max_blocks] int32
    cache_seqlens: torch.Tensor  # [B] int32
    page_block: int
    s_q: int
    h_q: int
    causal: bool
    softmax_scale: float

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.kv_rows.shape[0]) // self.page_block

    def kvcache_paged(self) -> torch.Tensor:
        """The cache viewed as [num_blocks, page_block, 1, d_k]."""
        return self.kv_rows.view(self.num_blocks, self.page_block, 1, self.kv_rows.shape[1])


def make_dense_case(seqlens: Sequence[int], s_q: int = 1, h_q: int = 128,
                    page_block: int = 64, dtype=torch.bfloat16, causal: bool = False,
                    seed: int = 0, spare_blocks: int = 0, shuffle: bool = True,
                    outlier_channels: int = 0, tail_fill: Optional[float] = None,
                    device="cpu", d_k: int = D_K) -> DenseCase:
    """A paged dense-decode problem.

    Pages: each request gets ceil(L/page_block) pages (at least one) plus
    ``spare_blocks`` unused pages overall; the physical order is a seeded
    random permutation (seed+1) unless ``shuffle`` is False. Unused table
    slots hold -1. ``tail_fill`` overwrites every cache row that no request
    can see (page tails beyond the length, spare pages) with that value, to
    check that masked rows never reach the result.
    """
    seqlens = np.asarray(seqlens, dtype=np.int64)
    B = len(seqlens)
    pages = np.maximum(1, -(-seqlens // page_block))
    total_pages = int(pages.sum()) + spare_blocks
    max_blocks = int(pages.max())
    perm = np.arange(total_pages)
    if shuffle:
        perm = np.random.default_rng(seed + 1).permutation(total_pages)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[cursor:cursor + pages[b]]
        cursor += pages[b]
    kv = make_latent_rows(total_pages * page_block, dtype=dtype, seed=seed,
                          outlier_channels=outlier_channels, device=device, d_k=d_k)
    if tail_fill is not None:
        visible = np.zeros(total_pages * page_block, dtype=bool)
        for b in range(B):
            visible[paged_rows_index(bt[b], int(seqlens[b]), page_block)] = True
        hidden = torch.from_numpy(~visible).to(kv.device)
        kv[hidden] = torch.tensor(tail_fill, dtype=dtype, device=kv.device)
    gq = _gen(seed + 10, device)
    q = torch.randn(B, s_q, h_q, d_k, generator=gq, device=device,
                    dtype=torch.float32).to(dtype)
    return DenseCase(q=q, kv_rows=kv, block_table=torch.from_numpy(bt),
                     cache_seqlens=torch.from_numpy(seqlens.astype(np.int32)),
                     page_block=page_block, s_q=s_q, h_q=h_q, causal=causal,
                     softmax_scale=d_k ** -0.5)


@dataclasses.dataclass
class SparseCase:
    q: torch.Tensor          # [B, s_q, h_q, 576] bf16
    kv_rows: torch.Tensor    # [B * tokens_per_request, 576] bf16 (pre-quantisation latent)
    indices: torch.Tensor    # [B, s_q, topk] int32, absolute row, -1 = invalid
    tokens_per_request: int
    page_block: int
    s_q: int
    h_q: int
    softmax_scale: float

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])


def make_sparse_case(batch: int, s_q: int, topk: int, tokens_per_request: int = 131072,
                     h_q: int = 128, page_block: int = 64, invalid_frac: float = 0.05,
                     seed: int = 0, outlier_channels: int = 0, device="cpu",
                     with_rows: bool = True, d_k: int = D_K) -> SparseCase:
    """Token-sparse decode: one contiguous cache of ``tokens_per_request`` rows
    per request (request b owns rows [b*T, (b+1)*T)); each query draws ``topk``
    distinct tokens of its request (seed+3) and exactly round(invalid_frac*topk)
    of its slots, at seeded random positions, are set to -1."""
    rng = np.random.default_rng(seed + 3)
    idx = np.empty((batch, s_q, topk), dtype=np.int32)
    n_bad = int(round(invalid_frac * topk))
    for b in range(batch):
        for i in range(s_q):
            sel = rng.choice(tokens_per_request, size=topk, replace=False)
            row = (sel + b * tokens_per_request).astype(np.int64)
            if n_bad:
                row[rng.choice(topk, size=n_bad, replace=False)] = -1
            idx[b, i] = row.astype(np.int32)
    rows = None
    if with_rows:
        rows = make_latent_rows(batch * tokens_per_request, dtype=torch.bfloat16, seed=seed,
                                outlier_channels=outlier_channels, device=device, d_k=d_k)
    gq = _gen(seed + 10, device)
    q = torch.randn(batch, s_q, h_q, d_k, generator=gq, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    return SparseCase(q=q, kv_rows=rows, indices=torch.from_numpy(idx),
                      tokens_per_request=tokens_per_request, page_block=page_block,
                      s_q=s_q, h_q=h_q, softmax_scale=d_k ** -0.5)


@dataclasses.dataclass
class AbsorbCase:
    """Per-head projection weights and activations around the decode kernel:
    q_nope [T, h, d_h], o_lat [T, h, d_c], w_uk and w_uv [h, d_h, d_c]."""
    q_nope: torch.Tensor
    o_lat: torch.Tensor
    w_uk: torch.Tensor
    w_uv: torch.Tensor


def make_absorb_case(tokens: int, h: int = 128, d_h: int = 128, d_c: int = 512, dtype=torch.bfloat16,
                     seed: int = 0, device="cpu") -> AbsorbCase:
    """Activations ~N(0,1); weights ~N(0, 1/fan_in) so that every output is ~N(0,1)
    (W^UK contracts over d_h, W^UV over d_c). Seeds seed+20 .. seed+23."""
    def rnd(shape, k, std):
        g = _gen(seed + 20 + k, device)
        return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)
    return AbsorbCase(q_nope=rnd((tokens, h, d_h), 0, 1.0), o_lat=rnd((tokens, h, d_c), 1, 1.0),
                      w_uk=rnd((h, d_h, d_c), 2, d_h ** -0.5), w_uv=rnd((h, d_h, d_c), 3, d_c ** -0.5))
