// decode_dense.cuh -- MLA decode over a paged BF16/FP16 latent cache, sm_103a.
//
// What one 2-CTA cluster computes. A persistent cluster owns one range of the
// split-KV schedule (a list of (virtual request, tile range) pieces). For a
// piece it keeps, for all 128 heads, the online-softmax state (m, l) and the
// 512-wide latent output O, and walks the piece's 64-token tiles:
//   S  = Q K^T              (128 heads x 64 tokens, contraction over 576)
//   P  = exp(S*scale - m)   (online softmax with running max / sum)
//   O += P V                (V = the first 512 dims of the same rows)
// ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §五 flashDecode, §六 absorbed MQA
// shape, §七 split-KV; "FlashMLA 实战", §最小调用).
//
// How the work is laid out on GB300. The fp32 O for 128 heads x 512 fills the
// whole 128-lane x 512-column tensor memory of one SM, so the two CTAs of the
// cluster split the latent dimension: CTA r keeps O[:, 256r : 256r+256] in TMEM
// (256 columns) and loads only its own 64-wide column chunks of Q and of every
// KV tile -- CTA 0 chunks {0,1,2,3} plus the RoPE chunk 8, CTA 1 chunks
// {4,5,6,7}. Each CTA computes a partial S over its chunks with single-CTA
// UMMA (M=128 heads, N=64 tokens); the two fp32 partials are exchanged through
// distributed shared memory and summed, so both CTAs hold the full S, run the
// same softmax (bit-identical), and accumulate P . V for their own half of the
// latent (M=128, N=256, K=64). No tensor-core work is duplicated and no KV byte
// is read twice. (Prior art on the pages: the Hopper kernel splits O between
// two warpgroups -- seesaw -- because the register file is full, and the FP8
// kernel pairs two CTAs over DSM -- Crossover; here the pair exists because
// TMEM is full.)
//
// Warp roles (256 threads): warp 0 lane 0 issues TMA loads; warp 1 owns TMEM
// and lane 0 issues UMMA; warps 4-7 are the softmax / exchange / epilogue
// warps, thread h <-> TMEM lane h <-> head h. Warps 2-3 only take part in
// set-up and tear-down.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "params.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace mla {
namespace dense {

constexpr int kNS = 2;                     // KV ring slots (tiles)
constexpr int kMaxChunks = 5;              // 64-wide column chunks per CTA
constexpr int kQChunk = 128 * 128;         // 128 rows x 64 x 2 B
constexpr int kKChunk = 64 * 128;          // 64 tokens x 64 x 2 B
constexpr int kSlot = kMaxChunks * kKChunk;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;            // S buffers at columns 256 and 320

// shared memory map (offsets from a 1024-B aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + kMaxChunks * kQChunk;
constexpr uint32_t OFF_P = OFF_RING + kNS * kSlot;
constexpr uint32_t OFF_SX = OFF_P + 128 * 128;          // 128 rows x 64 fp32
constexpr uint32_t OFF_BAR = OFF_SX + 128 * 256;
enum : uint32_t {
  B_FULL = 0, B_EMPTY = B_FULL + kNS, B_QFULL = B_EMPTY + kNS, B_QEMPTY, B_SFULL, B_SEMPTY = B_SFULL + 2,
  B_PFULL = B_SEMPTY + 2, B_PEMPTY, B_OEMPTY, B_XFULL, B_XEMPTY, B_DRAIN, B_COUNT
};
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;    // tmem slot, abort flag, ok flag
constexpr uint32_t kSmemBytes = OFF_MISC + 64 + 1024;   // + alignment slack

__device__ __forceinline__ int chunk_id(uint32_t rank, int ci) { return rank == 0 ? (ci < 4 ? ci : 8) : 4 + ci; }

// iteration over the pieces of one SM part (every role walks the same list)
struct PieceIter {
  const DecodeParams* p;
  int bv, bt, ev, et, first_split;
  int v;
  __device__ __forceinline__ PieceIter(const DecodeParams& prm, int part) : p(&prm) {
    const int32_t* r = prm.meta + H_WORDS + part * P_WORDS;
    bv = r[P_BV]; bt = r[P_BT]; ev = r[P_EV]; et = r[P_ET]; first_split = r[P_SPLIT];
    const int V = prm.batch * prm.s_q;
    if (bv < 0 || bv >= V || ev < bv || ev >= V) { bv = 0; ev = -1; }  // empty part
    v = bv - 1;
  }
  // advance to the next non-empty piece; false when done
  __device__ __forceinline__ bool next(int& vv, int& t0, int& t1, int& len, int& split, bool& fin) {
    while (++v <= ev) {
      const int n = vreq_tiles(p->seqlens, p->topk, p->batch, p->s_q, p->causal, v, &len);
      t0 = (v == bv) ? bt : 0;
      t1 = (v == ev) ? et : n;
      t0 = t0 < 0 ? 0 : t0;
      t1 = t1 > n ? n : t1;
      if (t1 <= t0) continue;
      const int ord = (v == bv) ? first_split : 0;
      const int off = p->split_off[v];
      const int ns = p->split_off[v + 1] - off;
      split = off + ord;
      fin = (ns == 1);
      vv = v;
      return true;
    }
    return false;
  }
};

template <bool kFp16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_dense_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                            const DecodeParams p) {
  using OutT = typename std::conditional<kFp16, __half, __nv_bfloat16>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int part = (int)cluster_id_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqc = rank == 0 ? 5 : 4;  // own column chunks

  auto bar = [&](uint32_t i) { return sb + OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* ok_flag = misc + 2;
  const Guard guard{abort_flag, p.status, 1500000000ull};

  const uint32_t fp = warp == 0 ? lengths_hash_warp(p.seqlens, p.batch, p.topk) : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SEMPTY + s), 128);
    }
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_PEMPTY), 1);
    mbar_init(bar(B_OEMPTY), 128);
    mbar_init(bar(B_XFULL), 128);
    mbar_init(bar(B_XEMPTY), 128);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0u;
    *ok_flag = metadata_matches(p, kTile, fp) ? 1u : 0u;
    if (!*ok_flag && rank == 0) atomicOr(p.status, STATUS_STALE);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool ok = *ok_flag != 0u;

  if (ok && warp == 0 && lane == 0) {
    // ---------------- producer: Q chunks per piece, KV chunks per tile ----------------
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kv);
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    PieceIter it(p, part);
    int v, t0, t1, len, split;
    bool fin;
    int g = 0, qn = 0;
    bool issued[kNS] = {};
    uint32_t last_par[kNS] = {};
    bool q_issued = false;
    uint32_t q_par = 0;
    while (it.next(v, t0, t1, len, split, fin)) {
      if (!wait(bar(B_QEMPTY), (qn & 1) ^ 1, guard)) break;
      const int b = v % p.batch, i = v / p.batch;
      const int qrow = (b * p.s_q + i) * 128;
      mbar_arrive_expect_tx(bar(B_QFULL), nqc * kQChunk);
      for (int ci = 0; ci < nqc; ++ci)
        tma_load_2d(sb + OFF_Q + ci * kQChunk, &tm_q, bar(B_QFULL), 64 * chunk_id(rank, ci), qrow, pol_q);
      q_issued = true;
      q_par = qn & 1;
      ++qn;
      bool stop = false;
      for (int t = t0; t < t1; ++t, ++g) {
        const int s = g % kNS;
        if (!wait(bar(B_EMPTY + s), ((g / kNS) & 1) ^ 1, guard)) { stop = true; break; }
        int page = t < p.max_blocks ? p.block_table[(int64_t)b * p.max_blocks + t] : -1;
        if (page < 0 || page >= p.num_blocks) page = 0;  // tile is masked by the softmax warps
        mbar_arrive_expect_tx(bar(B_FULL + s), nqc * kKChunk);
        for (int ci = 0; ci < nqc; ++ci)
          tma_load_2d(sb + OFF_RING + s * kSlot + ci * kKChunk, &tm_kv, bar(B_FULL + s), 64 * chunk_id(rank, ci),
                      page * kTile, pol_kv);
        issued[s] = true;
        last_par[s] = (g / kNS) & 1;
      }
      if (stop) break;
    }
    // never leave with a copy in flight into this CTA's shared memory
    for (int s = 0; s < kNS; ++s)
      if (issued[s]) {
        const uint64_t t_0 = globaltimer();
        while (!mbar_try_wait(bar(B_FULL + s), last_par[s]) && globaltimer() - t_0 < 200000000ull) {}
      }
    if (q_issued) {
      const uint64_t t_0 = globaltimer();
      while (!mbar_try_wait(bar(B_QFULL), q_par) && globaltimer() - t_0 < 200000000ull) {}
    }
  } else if (ok && warp == 1 && lane == 0) {
    // ---------------- UMMA issuer ----------------
    constexpr uint32_t idesc_qk = idesc_f16(128, 64, !kFp16, false, false);
    constexpr uint32_t idesc_pv = idesc_f16(128, 256, !kFp16, false, true);
    PieceIter it(p, part);
    int v, t0, t1, len, split;
    bool fin;
    int g = 0, qn = 0, piece = 0;
    int pend_g = -1, pend_piece = 0;
    bool pend_first = false, failed = false;
    auto issue_pv = [&](int gp, bool first, int pc) -> bool {
      if (!wait(bar(B_PFULL), gp & 1, guard)) return false;
      if (first && pc > 0 && !wait(bar(B_OEMPTY), (pc - 1) & 1, guard)) return false;
      tc_fence_after();
      const uint32_t slot = sb + OFF_RING + (gp % kNS) * kSlot;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t a = sdesc_sw128(sb + OFF_P + 32 * k, 16, 1024);
        const uint64_t bdesc = sdesc_sw128(slot + k * 2048, kKChunk, 1024);  // MN-major V: 16 tokens per step
        umma_ss(tmem, a, bdesc, idesc_pv, (first && k == 0) ? 0u : 1u);
      }
      umma_commit(bar(B_PEMPTY));
      umma_commit(bar(B_EMPTY + gp % kNS));
      return true;
    };
    while (!failed && it.next(v, t0, t1, len, split, fin)) {
      if (!wait(bar(B_QFULL), qn & 1, guard)) break;
      ++qn;
      for (int t = t0; t < t1; ++t, ++g) {
        const int s = g % kNS, sbuf = g & 1;
        if (!wait(bar(B_FULL + s), (g / kNS) & 1, guard) ||
            !wait(bar(B_SEMPTY + sbuf), ((g >> 1) & 1) ^ 1, guard)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t slot = sb + OFF_RING + s * kSlot;
        const uint32_t dS = tmem + kColS + 64u * sbuf;
        for (int ci = 0; ci < nqc; ++ci) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = sdesc_sw128(sb + OFF_Q + ci * kQChunk + 32 * k, 16, 1024);
            const uint64_t bdesc = sdesc_sw128(slot + ci * kKChunk + 32 * k, 16, 1024);
            umma_ss(dS, a, bdesc, idesc_qk, (ci | k) ? 1u : 0u);
          }
        }
        umma_commit(bar(B_SFULL + sbuf));
        if (t == t1 - 1) umma_commit(bar(B_QEMPTY));
        if (pend_g >= 0 && !issue_pv(pend_g, pend_first, pend_piece)) {
          failed = true;
          break;
        }
        pend_g = g;
        pend_first = (t == t0);
        pend_piece = piece;
      }
      ++piece;
    }
    if (!failed && pend_g >= 0) issue_pv(pend_g, pend_first, pend_piece);
    // every UMMA issued above has completed before TMEM is released
    umma_commit(bar(B_DRAIN));
    const uint64_t t_0 = globaltimer();
    while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer() - t_0 < 200000000ull) {}
  } else if (ok && warp >= 4) {
    // ---------------- softmax / exchange / epilogue ----------------
    const int h = threadIdx.x - 128;                      // head = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp - 4)) << 16);
    const uint32_t x_local = sb + OFF_SX + h * 256;
    const uint32_t x_remote = mapa(x_local, peer);
    const uint32_t xfull_remote = mapa(bar(B_XFULL), peer);
    const uint32_t xempty_remote = mapa(bar(B_XEMPTY), peer);
    const uint32_t p_row = sb + OFF_P + (h >> 3) * 1024 + (h & 7) * 128;
    const float sl2 = p.scale_log2;
    PieceIter it(p, part);
    int v, t0, t1, len, split;
    bool fin;
    int g = 0;
    bool failed = false;
    while (!failed && it.next(v, t0, t1, len, split, fin)) {
      const int b = v % p.batch, i = v / p.batch;
      float m = -INFINITY, l = 0.f;
      for (int t = t0; t < t1; ++t, ++g) {
        const int sbuf = g & 1;
        uint32_t sr[64];
        if (!__all_sync(0xffffffffu, wait(bar(B_SFULL + sbuf), (g >> 1) & 1, guard))) { failed = true; break; }
        tc_fence_after();
        tmem_ld32(tl + kColS + 64u * sbuf, sr);
        tmem_ld32(tl + kColS + 64u * sbuf + 32u, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(B_SEMPTY + sbuf));
        // send my partial scores to the peer, receive and add the peer's
        if (!__all_sync(0xffffffffu, wait_cluster(bar(B_XEMPTY), (g & 1) ^ 1, guard))) { failed = true; break; }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          st_cluster_v4(x_remote + ((u ^ (h & 7)) << 4), __uint_as_float(sr[4 * u]), __uint_as_float(sr[4 * u + 1]),
                        __uint_as_float(sr[4 * u + 2]), __uint_as_float(sr[4 * u + 3]));
        mbar_arrive_remote(xfull_remote);
        if (!__all_sync(0xffffffffu, wait_cluster(bar(B_XFULL), g & 1, guard))) { failed = true; break; }
        float s[64];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float4 o = ld_shared_v4f(x_local + ((u ^ (h & 7)) << 4));
          s[4 * u + 0] = __uint_as_float(sr[4 * u + 0]) + o.x;
          s[4 * u + 1] = __uint_as_float(sr[4 * u + 1]) + o.y;
          s[4 * u + 2] = __uint_as_float(sr[4 * u + 2]) + o.z;
          s[4 * u + 3] = __uint_as_float(sr[4 * u + 3]) + o.w;
        }
        mbar_arrive_remote(xempty_remote);
        // valid tokens of this tile (a bad page masks the whole tile)
        int nv = len - t * kTile;
        nv = nv > kTile ? kTile : nv;
        {
          const int page = t < p.max_blocks ? p.block_table[(int64_t)b * p.max_blocks + t] : -1;
          if (page < 0 || page >= p.num_blocks) {
            if (h == 0 && rank == 0) atomicOr(p.status, STATUS_INDEX);
            nv = 0;
          }
        }
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          s[k] = k < nv ? s[k] * sl2 : -INFINITY;
          mt = fmaxf(mt, s[k]);
        }
        const float m_new = fmaxf(m, mt);
        // lazy rescale: keep the old reference max unless the new one is
        // more than 2^8 larger (P stays <= 256, exact in the accumulation)
        const bool resc = m_new > m + 8.0f;
        const float m_use = resc ? m_new : m;
        const float alpha = resc ? exp2_approx(m - m_new) : 1.0f;
        const float m_ref = m_use == -INFINITY ? 0.f : m_use;
        float rs = 0.f;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          s[k] = exp2_approx(s[k] - m_ref);
          rs += s[k];
        }
        l = l * alpha + rs;
        m = m_use;
        // the previous P . V has finished: P buffer and O are free
        if (g > 0 && !__all_sync(0xffffffffu, wait(bar(B_PEMPTY), (g - 1) & 1, guard))) { failed = true; break; }
        tc_fence_after();
        if (resc && t != t0) {
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tmem_ld32(tl + 32u * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(tl + 32u * c, r);
          }
          tmem_wait_st();
        }
        if (nv < kTile) {
          // zero the V rows of masked tokens: 0 * (whatever is there) must not
          // turn into NaN inside P . V
          const uint32_t slot = sb + OFF_RING + (g % kNS) * kSlot;
          const int nrow = (kTile - nv) * 4;  // rows x 4 V chunks
          for (int e = h; e < nrow * 8; e += 128) {
            const int rr = e >> 3, ch = rr / (kTile - nv), row = nv + rr % (kTile - nv);
            st_shared_v4(slot + ch * kKChunk + row * 128 + (e & 7) * 16, 0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t w0 = kFp16 ? pack_f16x2(s[8 * u + 0], s[8 * u + 1]) : pack_bf16x2(s[8 * u + 0], s[8 * u + 1]);
          const uint32_t w1 = kFp16 ? pack_f16x2(s[8 * u + 2], s[8 * u + 3]) : pack_bf16x2(s[8 * u + 2], s[8 * u + 3]);
          const uint32_t w2 = kFp16 ? pack_f16x2(s[8 * u + 4], s[8 * u + 5]) : pack_bf16x2(s[8 * u + 4], s[8 * u + 5]);
          const uint32_t w3 = kFp16 ? pack_f16x2(s[8 * u + 6], s[8 * u + 7]) : pack_bf16x2(s[8 * u + 6], s[8 * u + 7]);
          st_shared_v4(p_row + ((u ^ (h & 7)) << 4), w0, w1, w2, w3);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
      }
      if (failed) break;
      // ---- epilogue of the piece: O / l -> out (single piece) or partial ----
      if (!__all_sync(0xffffffffu, wait(bar(B_PEMPTY), (g - 1) & 1, guard))) { failed = true; break; }
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      const int64_t row = (int64_t)(b * p.s_q + i) * 128 + h;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32u * c, r);
        tmem_wait_ld();
        if (fin) {
          OutT* dst = reinterpret_cast<OutT*>(p.out) + row * kDV + 256 * rank + 32 * c;
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 w;
            const float* f = reinterpret_cast<const float*>(r + k);
            w.x = kFp16 ? pack_f16x2(f[0] * inv_l, f[1] * inv_l) : pack_bf16x2(f[0] * inv_l, f[1] * inv_l);
            w.y = kFp16 ? pack_f16x2(f[2] * inv_l, f[3] * inv_l) : pack_bf16x2(f[2] * inv_l, f[3] * inv_l);
            w.z = kFp16 ? pack_f16x2(f[4] * inv_l, f[5] * inv_l) : pack_bf16x2(f[4] * inv_l, f[5] * inv_l);
            w.w = kFp16 ? pack_f16x2(f[6] * inv_l, f[7] * inv_l) : pack_bf16x2(f[6] * inv_l, f[7] * inv_l);
            *reinterpret_cast<uint4*>(dst + k) = w;
          }
        } else {
          float* dst = p.o_part + ((int64_t)split * 128 + h) * kDV + 256 * rank + 32 * c;
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + k) =
                make_float4(__uint_as_float(r[k]) * inv_l, __uint_as_float(r[k + 1]) * inv_l,
                            __uint_as_float(r[k + 2]) * inv_l, __uint_as_float(r[k + 3]) * inv_l);
        }
      }
      if (rank == 0) {
        if (fin) p.lse[row] = lse;
        else p.lse_part[(int64_t)split * 128 + h] = lse;
      }
      tc_fence_before();
      mbar_arrive(bar(B_OEMPTY));
    }
  }

  // ---------------- tear-down ----------------
  __syncwarp();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace dense
}  // namespace mla
