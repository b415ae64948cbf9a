// decode_fewheads.cuh -- MLA decode with few query heads (h_q = 16) over a
// paged BF16/FP16 latent cache, sm_103a.
//
// With 16 heads the heads cannot fill the M dimension of a UMMA, so the tile
// is transposed (the formulation of the FlashMLA-ETAP page, §2.2 and §3.2):
// tokens become M and heads N.
//   S^T = K Q^T        (64 tokens x 16 heads, contraction over all 576 dims)
//   P^T = softmax over the tokens of each head column (online, running max/sum)
//   O^T += V^T P^T     (512 dims x 16 heads, as four 128-dim blocks)
// and the epilogue writes O^T / l transposed back into [head][dim] order.
// The work is bound by the cache bytes (about 30 FLOP per byte), so one CTA
// per SM streams 64-token tiles; no pairing is needed because O^T is only 64
// TMEM columns. A tile's turnaround (its slot freed by a P . V, the copy, the
// S^T MMAs, the softmax, its own P . V) is shared by the tiles in flight, so
// the ring is cut finer than a 72 KB tile: 11 units of two latent chunks
// (16 KB, the V^T block of 128 dims that one P . V MMA reads) and 3 RoPE
// chunks (8 KB, read only by S^T and freed as soon as it completes), 2.75
// tiles in all, where two whole-tile slots are all that fit beside Q and P.
// S^T multiplies each unit as soon as it lands, so only the last pair of a
// tile (whose unit the P . V two tiles back frees) is on the turnaround.
//
// Memory map. TMEM (128 columns): S^T buffers [0,16) and [16,32), O^T blocks
// [64 + 16j, 80 + 16j) for dims [128j, 128j+128). Shared memory: the unit ring
// (chunks of 64 dims x 64 tokens, 128-B swizzled; tile g's latent pair j is
// unit (4g + j) mod 11, its RoPE chunk unit g mod 3), Q of the piece (9 chunks
// of 64 dims x 16 heads), two P^T buffers ([16 heads][64 tokens], 128-B
// swizzled), reduction scratch.
//
// Warp roles (224 threads): warp 0 lane 0 issues TMA; warp 1 owns TMEM and lane
// 0 issues S^T; lane 0 of warp 6 issues P . V; warps 2-5 are the softmax
// warps, warp w serving TMEM lanes 32*(w%4) .. +31. An M=64 accumulator keeps
// its rows in lanes 0-15 of each 32-lane quarter, so softmax thread (quarter
// q, lane < 16) holds token 16q + lane of the tile with its 16 head scores;
// for the 128-row O^T blocks every lane is one output dim.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "params.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace mla {
namespace few {

constexpr int kNH = 16;                       // heads
constexpr int kThreads = 224;
constexpr int kSoftWarps = 4;                 // warps 2-5
constexpr int kPvWarp = 6;                    // its lane 0 issues P . V
constexpr int kChunks = 9;                    // 576 = 9 x 64 dims
constexpr uint32_t kChunkBytes = 64 * 128;    // 64 tokens x 64 dims x 2 B
constexpr uint32_t kQChunk = kNH * 128;       // 16 heads x 64 dims x 2 B
constexpr uint32_t kQBytes = kChunks * kQChunk;
constexpr uint32_t kPBytes = kNH * 128;       // [16 heads][64 tokens] x 2 B
constexpr int kPairs = 11;                    // ring units of two latent chunks (16 KB)
constexpr int kRopes = 3;                     // ring units of one RoPE chunk (8 KB)
constexpr uint32_t kPairBytes = 2 * kChunkBytes;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColO = 64;
constexpr uint32_t kSoftBar = 1;              // named barrier of the 128 softmax threads

constexpr uint32_t OFF_RING = 0;
constexpr uint32_t OFF_ROPE = OFF_RING + kPairs * kPairBytes;
constexpr uint32_t OFF_Q = OFF_ROPE + kRopes * kChunkBytes;
constexpr uint32_t OFF_P = OFF_Q + kQBytes;
constexpr uint32_t OFF_RED = OFF_P + 2 * kPBytes;          // [4 warps][16 heads] floats
constexpr uint32_t OFF_BAR = OFF_RED + kSoftWarps * kNH * 4;
enum : uint32_t {
  B_FULL = 0, B_EMPTY = B_FULL + kPairs, B_RFULL = B_EMPTY + kPairs, B_REMPTY = B_RFULL + kRopes,
  B_QFULL = B_REMPTY + kRopes, B_QEMPTY = B_QFULL + 1, B_SFULL = B_QEMPTY + 1,
  B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2, B_PEMPTY = B_PFULL + 2, B_OEMPTY = B_PEMPTY + 2,
  B_DRAIN = B_OEMPTY + 1, B_DRAIN2 = B_DRAIN + 1, B_STALL = B_DRAIN2 + 1, B_COUNT = B_STALL + 1
};
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;
constexpr uint32_t kSmemBytes = OFF_MISC + 64 + 1024;
static_assert(OFF_ROPE % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_P % 1024 == 0,
              "128-B swizzled operands need 1024-B alignment");
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }
// ring unit n (n = 4g + j: latent chunks 2j, 2j+1 of tile g)
__device__ __forceinline__ uint32_t pair_addr(uint32_t sb, int n) {
  return sb + OFF_RING + (uint32_t)(n % kPairs) * kPairBytes;
}
// chunk c (0..8, 8 = RoPE) of tile g
__device__ __forceinline__ uint32_t chunk_addr(uint32_t sb, int g, int c) {
  return c < 8 ? pair_addr(sb, 4 * g + (c >> 1)) + (uint32_t)(c & 1) * kChunkBytes
               : sb + OFF_ROPE + (uint32_t)(g % kRopes) * kChunkBytes;
}

template <bool kFp16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_fewheads_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k2,
                               const __grid_constant__ CUtensorMap tm_k1, const DecodeParams p) {
  using OutT = typename std::conditional<kFp16, __half, __nv_bfloat16>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int part = (int)blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](uint32_t i) { return sb + OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* ok_flag = misc + 2;
  const Guard guard{abort_flag, p.status, kWaitLimitCycles};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairs; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int s = 0; s < kRopes; ++s) {
      mbar_init(bar(B_RFULL + s), 1);
      mbar_init(bar(B_REMPTY + s), 1);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SEMPTY + s), kSoftWarps);
      mbar_init(bar(B_PFULL + s), kSoftWarps);
      mbar_init(bar(B_PEMPTY + s), 1);
    }
    mbar_init(bar(B_OEMPTY), kSoftWarps);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN2), 1);
    mbar_init(bar(B_STALL), 1);
    *abort_flag = 0u;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  // nothing above reads global memory; wait for the kernels this one depends
  // on (programmatic dependent launch) before the first read. The metadata
  // header is loaded before the lengths are hashed, so that both reads are in
  // flight together.
  pdl_wait();
  int32_t hdr[H_WORDS];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < H_WORDS; ++w) hdr[w] = p.meta[w];
  }
  const uint32_t fp = warp == 0 ? lengths_hash_warp(p.seqlens, p.batch, p.topk) : 0u;
  if (threadIdx.x == 0) {
    *ok_flag = header_matches(hdr, p, kTile, fp) ? 1u : 0u;
    if (!*ok_flag) atomicOr(p.status, STATUS_STALE);
    fence_mbar_init();
    if (*ok_flag && p.stall_cycles) {
      // test hook: a bounded wait on a barrier nothing arrives at gives up
      // and reports STATUS_TIMEOUT before anything is issued
      const Guard g_stall{abort_flag, p.status, p.stall_cycles};
      if (!wait(bar(B_STALL), 0, g_stall)) *ok_flag = 0u;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool ok = *ok_flag != 0u;

  if (ok && warp == 0 && lane == 0) {
    // ---------------- producer: Q per piece; per tile four latent pairs and the RoPE chunk ----------------
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k2);
    prefetch_tmap(&tm_k1);
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    PieceIter it(p, part);
    Piece pc;
    int g = 0, qn = 0, q_last = -1;
    int last_n[kPairs], last_r[kRopes];
    for (int u = 0; u < kPairs; ++u) last_n[u] = -1;
    for (int u = 0; u < kRopes; ++u) last_r[u] = -1;
    bool stop = false;
    auto raw_page = [&](int b, int t) {
      return t < p.max_blocks ? __ldg(p.block_table + (int64_t)b * p.max_blocks + t) : -1;
    };
    // the part's first block-table entry, read together with its first piece's
    // own loads (the part's range is checked, so the entry is in bounds)
    const int pre_v = it.v + 1, pre_t = it.bt < 0 ? 0 : it.bt;
    const int pre_pg = it.ev >= pre_v ? raw_page(pre_v % p.batch, pre_t) : -1;
    while (!stop && it.next(pc)) {
      const int b = pc.v % p.batch, i = pc.v / p.batch;
      if (!wait(bar(B_QEMPTY), (qn & 1) ^ 1, guard)) break;
      mbar_arrive_expect_tx(bar(B_QFULL), kQBytes);
      tma_load_3d(sb + OFF_Q, &tm_q, bar(B_QFULL), 0, (b * p.s_q + i) * kNH, 0, pol_q);
      q_last = qn++;
      // block-table entries are loaded one tile ahead
      int pg_next = (g == 0 && pc.v == pre_v && pc.t0 == pre_t) ? pre_pg : raw_page(b, pc.t0);
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        int page = pg_next;
        page = (page < 0 || page >= p.num_blocks) ? 0 : page;  // a bad page is masked by the softmax warps
        pg_next = raw_page(b, t + 1);
        // in the order the units free up: the RoPE chunk (freed by S^T three
        // tiles back), then latent pairs 0-2 (P . V three tiles back) and 3
        // (P . V two tiles back)
        const int r = g % kRopes;
        if (!wait(bar(B_REMPTY + r), ((g / kRopes) & 1) ^ 1, guard)) { stop = true; break; }
        mbar_arrive_expect_tx(bar(B_RFULL + r), kChunkBytes);
        tma_load_3d(sb + OFF_ROPE + r * kChunkBytes, &tm_k1, bar(B_RFULL + r), 0, page * kTile, 8, pol_kv);
        last_r[r] = g;
        for (int j = 0; j < 4 && !stop; ++j) {  // latent chunks 2j, 2j+1: one 16 KB box
          const int n = 4 * g + j, u = n % kPairs;
          if (!wait(bar(B_EMPTY + u), ((n / kPairs) & 1) ^ 1, guard)) { stop = true; break; }
          mbar_arrive_expect_tx(bar(B_FULL + u), kPairBytes);
          tma_load_3d(sb + OFF_RING + u * kPairBytes, &tm_k2, bar(B_FULL + u), 0, page * kTile, 2 * j, pol_kv);
          last_n[u] = n;
        }
        if (stop) break;
      }
    }
    // never leave with a copy in flight into this CTA's shared memory
    for (int u = 0; u < kPairs; ++u)
      if (last_n[u] >= 0) {
        const uint64_t t_0 = cycles();
        while (!mbar_try_wait(bar(B_FULL + u), (last_n[u] / kPairs) & 1) && cycles() - t_0 < kDrainLimitCycles) {}
      }
    for (int u = 0; u < kRopes; ++u)
      if (last_r[u] >= 0) {
        const uint64_t t_0 = cycles();
        while (!mbar_try_wait(bar(B_RFULL + u), (last_r[u] / kRopes) & 1) && cycles() - t_0 < kDrainLimitCycles) {}
      }
    if (q_last >= 0) {
      const uint64_t t_0 = cycles();
      while (!mbar_try_wait(bar(B_QFULL), q_last & 1) && cycles() - t_0 < kDrainLimitCycles) {}
    }
  } else if (ok && lane == 0 && (warp == 1 || warp == kPvWarp)) {
    // ---------------- UMMA issue: S^T by warp 1, P . V by warp kPvWarp ----------------
    // Two issuing threads, each waiting only on its own inputs, so that a
    // ready P . V never waits behind the issue of a tile's 36 S^T MMAs.
    constexpr uint32_t idesc_qk = idesc_f16(64, kNH, !kFp16, false, false);   // K tile (tokens x dims), Q (heads x dims)
    constexpr uint32_t idesc_pv = idesc_f16(128, kNH, !kFp16, true, false);   // V^T (dims-major), P^T (heads x tokens)
    PieceIter it(p, part);
    Piece pc;
    int g = 0, k = 0;
    bool failed = false;
    uint32_t drain_bar = bar(B_DRAIN);
    if (warp == 1) {
      while (!failed && it.next(pc)) {
        if (!wait(bar(B_QFULL), k & 1, guard)) break;
        for (int t = pc.t0; t < pc.t1; ++t, ++g) {
          const int sbuf = g & 1;
          // S^T accumulates chunk by chunk in any order: the RoPE chunk and
          // the latent pairs are each multiplied as soon as they have landed,
          // so that only the last pair's MMAs follow the last copy (that
          // pair's unit is freed by the P . V two tiles back, the others'
          // by the one three tiles back)
          if (!wait(bar(B_SEMPTY + sbuf), ((g >> 1) & 1) ^ 1, guard) ||
              !wait(bar(B_RFULL + g % kRopes), (g / kRopes) & 1, guard)) {
            failed = true;
            break;
          }
          tc_fence_after();
          auto issue_chunk = [&](int c, bool first) {
            const uint64_t d_k = sdesc_sw128(chunk_addr(sb, g, c), 16, 1024);
            const uint64_t d_q = sdesc_sw128(sb + OFF_Q + c * kQChunk, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss(tmem + 16u * sbuf, d_k + 2u * kk, d_q + 2u * kk, idesc_qk, (first && kk == 0) ? 0u : 1u);
          };
          issue_chunk(8, true);
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            const int n = 4 * g + j;
            if (!wait(bar(B_FULL + n % kPairs), (n / kPairs) & 1, guard)) {
              failed = true;
              break;
            }
            tc_fence_after();
            issue_chunk(2 * j, false);
            issue_chunk(2 * j + 1, false);
          }
          if (failed) break;
          umma_commit(bar(B_SFULL + sbuf));
          umma_commit(bar(B_REMPTY + g % kRopes));  // only S^T reads the RoPE chunk
        }
        if (failed) break;
        umma_commit(bar(B_QEMPTY));  // Q of the piece is free once its last S^T is done
        ++k;
      }
    } else {
      drain_bar = bar(B_DRAIN2);
      while (!failed && it.next(pc)) {
        for (int t = pc.t0; t < pc.t1; ++t, ++g) {
          // a piece's first P . V overwrites O^T: the previous piece's epilogue must have read it
          if (!wait(bar(B_PFULL + (g & 1)), (g >> 1) & 1, guard) ||
              (t == pc.t0 && k > 0 && !wait(bar(B_OEMPTY), (k - 1) & 1, guard))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const bool first = t == pc.t0;
          const uint64_t d_p = sdesc_sw128(sb + OFF_P + (g & 1) * kPBytes, 16, 1024);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // V^T block j: dims [128j, 128j+128) = chunks 2j, 2j+1 (one ring
            // unit, chunks 8 KB apart); +128 per 16 tokens
            const uint64_t d_v = sdesc_sw128(pair_addr(sb, 4 * g + j), kChunkBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss(tmem + kColO + 16u * j, d_v + 128u * kk, d_p + 2u * kk, idesc_pv, (first && kk == 0) ? 0u : 1u);
            // the unit is free once its block is done: pair 0's unit, freed
            // first, is the one that the last pair of tile g + 2 waits for
            umma_commit(bar(B_EMPTY + (4 * g + j) % kPairs));
          }
          umma_commit(bar(B_PEMPTY + (g & 1)));
        }
        ++k;
      }
    }
    // every UMMA this thread issued has completed before TMEM is released
    umma_commit(drain_bar);
    const uint64_t t_0 = cycles();
    while (!mbar_try_wait(drain_bar, 0) && cycles() - t_0 < kDrainLimitCycles) {}
  } else if (ok && warp >= 2 && warp < 2 + kSoftWarps) {
    // ---------------- softmax warps ----------------
    const int q4 = warp & 3;                              // TMEM lane quarter
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    const int tok = 16 * q4 + lane;                       // token of the tile held by this lane (lane < 16)
    const bool has_tok = lane < 16;
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    const float sl2 = p.scale_log2;
    // The 128 threads cross named barriers, so every failure is agreed on at
    // the next barrier (an OR over all threads) and they leave together.
    PieceIter it(p, part);
    Piece pc;
    int g = 0;
    bool failed = false;
    while (!failed && it.next(pc)) {
      const int b = pc.v % p.batch, i = pc.v / p.batch;
      MaskStream<false> ms;
      ms.start(p, pc);
      float m[kNH], l[kNH];   // running max (log2 domain, shared by all threads), this thread's share of the sum
#pragma unroll
      for (int h = 0; h < kNH; ++h) { m[h] = -INFINITY; l[h] = 0.f; }
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        const uint64_t vm = ms.next(p, t, warp == 2);
        const int sbuf = g & 1;
        bool okw = warp_all(!failed) && warp_all(wait(bar(B_SFULL + sbuf), (g >> 1) & 1, guard));
        float x[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) x[h] = -INFINITY;
        if (okw) {
          tc_fence_after();
          uint32_t r[kNH];
          tmem_ld16(tl + 16u * sbuf, r);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_SEMPTY + sbuf));
          if (has_tok && ((vm >> tok) & 1ull)) {
#pragma unroll
            for (int h = 0; h < kNH; ++h) x[h] = __uint_as_float(r[h]);
          }
        }
        // The reference max m of a head moves only when a score exceeds it
        // by more than 2^8 (so P <= 256). Each thread checks its own token's
        // scores; only when one of the 128 finds one above m + 8 (always on a
        // piece's first tile, where m is -inf) are the tile maxima exchanged,
        // and the result is what the exchange on every tile would give.
        bool over = false;
#pragma unroll
        for (int h = 0; h < kNH; ++h) over |= x[h] * sl2 > m[h] + 8.0f;
        // P^T[g&1] is free once P . V of tile g-2 is done; a wait that gave
        // up is agreed on at the vote below
        if (okw) okw = warp_all(wait(bar(B_PEMPTY + sbuf), ((g >> 1) & 1) ^ 1, guard));
        bool resc_any = false;
        float alpha[kNH], mu[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) { alpha[h] = 1.0f; mu[h] = m[h]; }
        if (named_sync_or(kSoftBar, 128, over || !okw)) {
          // tile max of every head: over the 16 token lanes, then over the 4 warps
          float mx[kNH];
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            float v = x[h];
#pragma unroll
            for (int o = 8; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            mx[h] = v;
          }
          if (lane < kNH) {
            float mine = mx[0];
#pragma unroll
            for (int h = 1; h < kNH; ++h) mine = lane == h ? mx[h] : mine;
            red[q4 * kNH + lane] = mine;
          }
          if (named_sync_or(kSoftBar, 128, !okw)) { failed = true; break; }
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float mt = fmaxf(fmaxf(red[h], red[kNH + h]), fmaxf(red[2 * kNH + h], red[3 * kNH + h])) * sl2;
            const float m_new = fmaxf(m[h], mt);
            const bool resc = m_new > m[h] + 8.0f;       // lazy rescale: P stays <= 2^8
            mu[h] = resc ? m_new : m[h];
            alpha[h] = resc ? exp2_approx(m[h] - m_new) : 1.0f;
            resc_any |= resc;
            m[h] = mu[h];
          }
        }
        // P^T of this tile; this thread's share of each head's sum
        uint32_t pk[kNH / 2];
#pragma unroll
        for (int h = 0; h < kNH; h += 2) {
          const float p0 = x[h] == -INFINITY ? 0.f : exp2_approx(fmaf(x[h], sl2, -mu[h]));
          const float p1 = x[h + 1] == -INFINITY ? 0.f : exp2_approx(fmaf(x[h + 1], sl2, -mu[h + 1]));
          l[h] = l[h] * alpha[h] + p0;
          l[h + 1] = l[h + 1] * alpha[h + 1] + p1;
          pk[h / 2] = kFp16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        }
        // a rescale of O^T needs every earlier P . V done (they complete in
        // order); resc_any is the same in every thread, and so is this barrier
        if (resc_any && t != pc.t0) {
          if (!warp_all(wait(bar(B_PEMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1, guard))) failed = true;
          if (warp_all(!failed)) {
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t o[kNH];
              tmem_ld16(tl + kColO + 16u * j, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kNH; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
              tmem_st16(tl + kColO + 16u * j, o);
            }
            tmem_wait_st();
          }
          if (named_sync_or(kSoftBar, 128, failed)) { failed = true; break; }
        }
        // masked tokens: zero their V rows (they may hold NaN; 0 * NaN would leak)
        if (vm != ~0ull) {
          for (int e = threadIdx.x - 64; e < 64 * 8 * 8; e += 128) {
            const int row = e >> 6, c = (e >> 3) & 7, u = e & 7;  // token, latent chunk, 16-B unit
            if (!((vm >> row) & 1ull)) st_shared_v4(chunk_addr(sb, g, c) + row * 128 + u * 16, 0u, 0u, 0u, 0u);
          }
        }
        if (has_tok) {
          // [head][token] with 16-B units of each 128-B head row swizzled by (head & 7)
          uint8_t* prow = smem + OFF_P + sbuf * kPBytes;
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const uint32_t off = h * 128 + ((((uint32_t)tok >> 3) ^ (uint32_t)(h & 7)) << 4) + (tok & 7) * 2;
            const uint32_t w = pk[h / 2];
            *reinterpret_cast<uint16_t*>(prow + off) = (uint16_t)((h & 1) ? (w >> 16) : (w & 0xFFFFu));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + sbuf));
      }
      if (failed) break;
      // ---- epilogue: l over the 64 token lanes, O^T / l -> out or partial ----
      float lt[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        float v = l[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        lt[h] = v;
      }
      bool okw = warp_all(wait(bar(B_PEMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1, guard));
      if (named_sync_or(kSoftBar, 128, !okw)) { failed = true; break; }  // every warp has read red[]
      if (lane < kNH) {
        float mine = lt[0];
#pragma unroll
        for (int h = 1; h < kNH; ++h) mine = lane == h ? lt[h] : mine;
        red[q4 * kNH + lane] = mine;
      }
      named_sync_na(kSoftBar, 128);
      float inv[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        const float L = red[h] + red[kNH + h] + red[2 * kNH + h] + red[3 * kNH + h];
        inv[h] = L > 0.f ? 1.0f / L : 0.f;
        lt[h] = L;
      }
      tc_fence_after();
      const int64_t row0 = (int64_t)(b * p.s_q + i) * kNH;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t o[kNH];
        tmem_ld16(tl + kColO + 16u * j, o);
        tmem_wait_ld();
        const int d = 128 * j + 32 * q4 + lane;
        if (pc.fin) {
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float v = __uint_as_float(o[h]) * inv[h];
            reinterpret_cast<OutT*>(p.out)[(row0 + h) * kDV + d] =
                kFp16 ? OutT(__float2half_rn(v)) : OutT(__float2bfloat16_rn(v));
          }
        } else {
#pragma unroll
          for (int h = 0; h < kNH; ++h)
            p.o_part[opart_index(pc.split, kNH, h, d)] = __uint_as_float(o[h]) * inv[h];
        }
      }
      if (warp == 2 && lane < kNH) {
        float Lh = lt[0], mh = m[0];
#pragma unroll
        for (int h = 1; h < kNH; ++h) {
          Lh = lane == h ? lt[h] : Lh;
          mh = lane == h ? m[h] : mh;
        }
        const float lse = Lh > 0.f ? (mh + log2f(Lh)) * 0.69314718055994530942f : -INFINITY;
        if (pc.fin) p.lse[row0 + lane] = lse;
        else p.lse_part[(int64_t)pc.split * kNH + lane] = lse;
      }
      tc_fence_before();
      named_sync_na(kSoftBar, 128);  // red[] is read before the next piece writes it
      if (lane == 0) mbar_arrive(bar(B_OEMPTY));
    }
  }

  // ---------------- tear-down ----------------
  __syncwarp();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace few
}  // namespace mla
