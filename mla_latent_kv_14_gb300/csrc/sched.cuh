// sched.cuh -- split-KV work schedule and the split combine.
//
// Schedule ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §七 'split-KV'):
// the (request, query-position) pairs are cut into 64-token tiles; the tile
// list, with a fixed cost per piece, is cut into `parts` contiguous ranges of
// nearly equal cost, one per persistent 2-CTA cluster. A request cut by a
// range boundary becomes several pieces whose partial (o, lse) the combine
// merges: m = max lse_i, o = sum o_i e^{lse_i - m} / sum e^{lse_i - m}
// (same section, the merge formula of online softmax).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "params.h"
#include "ptx.cuh"

namespace mla {

// visible tokens and tiles of virtual request v = i*batch + b
__device__ __forceinline__ int vreq_tiles(const int32_t* seqlens, int topk, int batch, int s_q, int causal,
                                          int v, int* len_out) {
  int L;
  if (topk > 0) {
    L = topk;
  } else {
    const int b = v % batch, i = v / batch;
    L = seqlens[b];
    if (causal) L = L - s_q + 1 + i;
  }
  L = L < 0 ? 0 : L;
  *len_out = L;
  return (L + kTile - 1) / kTile;
}

// Fingerprint of the per-request lengths (or of topk) baked into the
// metadata; a sum of mixed (index, length) words, so one warp computes it in
// parallel. Every lane of the calling warp must call it; all get the result.
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return x;
}
__device__ __forceinline__ uint32_t lengths_hash_warp(const int32_t* seqlens, int batch, int topk) {
  const int lane = threadIdx.x & 31;
  uint32_t h = 0;
  if (topk > 0) {
    h = lane == 0 ? mix32((uint32_t)topk ^ 0xA5A5A5A5u) : 0u;
  } else {
    for (int b = lane; b < batch; b += 32) h += mix32((uint32_t)seqlens[b] * 0x9E3779B1u + mix32((uint32_t)b));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
  return h ^ (uint32_t)batch;
}

constexpr int kMetaThreads = 1024;
constexpr int kMaxVreq = 8192;   // virtual requests the schedule kernel holds in shared memory

// block-wide exclusive scan of one int64 per thread; returns the block total
__device__ __forceinline__ long long block_exclusive_scan(long long x, long long* warp_tot, long long& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
    long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;          // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi; // block total
  }
  __syncthreads();
  excl = inc - x + warp_tot[warp];
  const long long tot = warp_tot[32];
  __syncthreads();
  return tot;
}

// The schedule as a closed form, computed by one block:
//  * request v costs n_v + ov (0 if it has no tile), ov = kPieceOverhead
//    (kPieceOverheadFewHeads for 16 heads); C_v is the exclusive prefix sum
//    of the costs and `total` their sum;
//  * part p owns the cost interval [p*per, (p+1)*per), per = ceil(total/parts)
//    (at least ov + 1); position x maps to the tile cursor
//    (v, max(0, x - C_v - ov)) of the request whose cost interval
//    holds x, so a part runs from cursor(p*per) to cursor((p+1)*per);
//  * a request is cut once per part boundary that falls on one of its tiles
//    other than its first.
__global__ void __launch_bounds__(kMetaThreads) mla_metadata_kernel(MetaParams p) {
  pdl_launch_dependents();  // the decode may start its set-up now; it waits for this grid before reading
  // This grid may itself be launched early, behind the previous call's
  // combine, which still reads the buffers written here: wait for it (and for
  // whatever produced the lengths) before the first global access.
  pdl_wait();
  extern __shared__ long long sh[];
  const int V = p.batch * p.s_q;
  long long* C = sh;                                        // [V + 1]
  int* n = reinterpret_cast<int*>(C + V + 1);               // [V]
  int* nsplit = n + V;                                      // [V]
  int* firstp = nsplit + V;                                 // [V]
  __shared__ long long warp_tot[33];
  __shared__ long long carry;
  const int ov = p.h_q == 128 ? kPieceOverhead : kPieceOverheadFewHeads;
  if (threadIdx.x == 0) carry = 0;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    int L;
    n[v] = vreq_tiles(p.seqlens, p.topk, p.batch, p.s_q, p.causal, v, &L);
    nsplit[v] = 0;
    firstp[v] = 0x7fffffff;
  }
  __syncthreads();
  for (int base = 0; base < V; base += blockDim.x) {
    const int v = base + threadIdx.x;
    const long long c = v < V && n[v] ? (long long)n[v] + ov : 0;
    long long excl;
    const long long tot = block_exclusive_scan(c, warp_tot, excl);
    if (v < V) C[v] = carry + excl;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
  const long long total = carry;
  if (threadIdx.x == 0) C[V] = total;
  __syncthreads();
  long long per = total > 0 ? (total + p.parts - 1) / p.parts : 1;
  if (per < ov + 1) per = ov + 1;
  auto cursor = [&](long long x, int& cv, int& ct) {
    if (x >= total) { cv = V; ct = 0; return; }
    int lo = 0, hi = V - 1;                 // largest v with C[v] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (C[mid] <= x) lo = mid; else hi = mid - 1;
    }
    cv = lo;
    const long long t = x - C[lo] - ov;
    ct = t > 0 ? (int)t : 0;
  };
  // part boundaries that cut a request
  for (int q = 1 + threadIdx.x; q < p.parts; q += blockDim.x) {
    int cv, ct;
    const long long x = (long long)q * per;
    cursor(x < total ? x : total, cv, ct);
    if (cv < V && ct > 0) {
      atomicAdd(&nsplit[cv], 1);
      atomicMin(&firstp[cv], q);
    }
  }
  __syncthreads();
  // pieces per request -> exclusive prefix (num_splits)
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < V; base += blockDim.x) {
    const int v = base + threadIdx.x;
    const long long c = v < V ? (long long)((n[v] ? 1 : 0) + nsplit[v]) : 0;
    long long excl;
    const long long tot = block_exclusive_scan(c, warp_tot, excl);
    if (v < V) p.split_off[v] = (int32_t)(carry + excl);
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.split_off[V] = (int32_t)carry;
  // part records
  int32_t* rec0 = p.meta + H_WORDS;
  for (int q = threadIdx.x; q < p.parts; q += blockDim.x) {
    int bv, bt, ve, te;
    const long long x0 = (long long)q * per, x1 = (long long)(q + 1) * per;
    cursor(x0 < total ? x0 : total, bv, bt);
    cursor(x1 < total ? x1 : total, ve, te);
    int32_t* r = rec0 + q * P_WORDS;
    if (bv >= V || (bv == ve && bt == te)) {
      r[P_BV] = -1;
      r[P_BT] = r[P_EV] = r[P_ET] = r[P_SPLIT] = 0;
    } else {
      r[P_BV] = bv;
      r[P_BT] = bt;
      r[P_EV] = te > 0 ? ve : ve - 1;
      r[P_ET] = te > 0 ? te : 0x7fffffff;
      r[P_SPLIT] = bt > 0 ? q - firstp[bv] + 1 : 0;
    }
  }
  const uint32_t fp = threadIdx.x < 32 ? lengths_hash_warp(p.seqlens, p.batch, p.topk) : 0u;
  if (threadIdx.x == 0) {
    int32_t* h = p.meta;
    h[H_MAGIC] = kMetaMagic;
    h[H_BATCH] = p.batch;
    h[H_SQ] = p.s_q;
    h[H_HQ] = p.h_q;
    h[H_TOPK] = p.topk;
    h[H_KVFMT] = p.kv_format;
    h[H_CAUSAL] = p.causal;
    h[H_PAGE] = p.page_block;
    h[H_PARTS] = p.parts;
    h[H_HASH] = (int32_t)fp;
    h[H_NPIECES] = (int32_t)carry;
    h[H_VREQ] = V;
  }
}

__host__ __device__ inline size_t metadata_smem_bytes(int vreq) {
  return (size_t)(vreq + 1) * sizeof(long long) + (size_t)vreq * 3 * sizeof(int);
}

// True when the metadata was built for exactly this call. `h` is its header,
// already loaded into registers (all comparisons evaluated, so the loads can
// all be in flight together); `fp` is the lengths fingerprint of this call
// (lengths_hash_warp).
__device__ __forceinline__ bool header_matches(const int32_t (&h)[H_WORDS], const DecodeParams& p, int page_block,
                                               uint32_t fp) {
  return (h[H_MAGIC] == kMetaMagic) & (h[H_BATCH] == p.batch) & (h[H_SQ] == p.s_q) & (h[H_HQ] == p.h_q) &
         (h[H_TOPK] == p.topk) & (h[H_KVFMT] == p.kv_format) & (h[H_CAUSAL] == p.causal) & (h[H_PAGE] == page_block) &
         (h[H_PARTS] == p.parts) & (h[H_VREQ] == p.batch * p.s_q) & ((uint32_t)h[H_HASH] == fp);
}

// Iteration over the pieces of one SM part: every role of a decode kernel
// walks the same list of (virtual request, tile range) pieces.
struct Piece {
  int v, t0, t1, len, split;
  bool fin;
};
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
  __device__ __forceinline__ bool next(Piece& pc) {
    while (++v <= ev) {
      int len;
      const int n = vreq_tiles(p->seqlens, p->topk, p->batch, p->s_q, p->causal, v, &len);
      int t0 = (v == bv) ? bt : 0;
      int t1 = (v == ev) ? et : n;
      t0 = t0 < 0 ? 0 : t0;
      t1 = t1 > n ? n : t1;
      if (t1 <= t0) continue;
      const int ord = (v == bv) ? first_split : 0;
      const int off = p->split_off[v];
      const int ns = p->split_off[v + 1] - off;
      pc.v = v; pc.t0 = t0; pc.t1 = t1; pc.len = len; pc.split = off + ord; pc.fin = (ns == 1);
      return true;
    }
    return false;
  }
};

// Tile validity masks, computed by a whole warp, bit k = token 64t+k.
// Dense: the first min(len - 64t, 64) tokens, or none if the tile's page is
// out of range (reported). Sparse: the index-list entries in [0, num_rows);
// -1 is skipped silently, other out-of-range entries are reported.
// The global loads behind a mask (block-table entries, index-list entries) are
// issued well before the mask is needed: a dense stream loads the pages of 32
// tiles per warp-wide load, one block ahead; a sparse stream loads the indices
// of tile t+2 while tile t is processed.
__device__ __forceinline__ int load_pages32(const DecodeParams& p, int b, int t) {
  const int tt = t + (int)(threadIdx.x & 31);
  return tt < p.max_blocks ? __ldg(p.block_table + (int64_t)b * p.max_blocks + tt) : -1;
}
__device__ __forceinline__ uint64_t dense_mask(const DecodeParams& p, int page, int t, int len, bool report) {
  int nv = len - t * kTile;
  nv = nv > kTile ? kTile : nv;
  if (page < 0 || page >= p.num_blocks) {
    if (report && (threadIdx.x & 31) == 0) atomicOr(p.status, STATUS_INDEX);
    nv = 0;
  }
  return nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
}
__device__ __forceinline__ void sparse_fetch(const DecodeParams& p, int v, int t, int& i0, int& i1) {
  const int b = v % p.batch, i = v / p.batch;
  const int32_t* row = p.indices + (int64_t)(b * p.s_q + i) * p.topk;
  const int k = 64 * t + (int)(threadIdx.x & 31);
  i0 = k < p.topk ? __ldg(row + k) : -1;
  i1 = k + 32 < p.topk ? __ldg(row + k + 32) : -1;
}
__device__ __forceinline__ uint64_t sparse_mask(const DecodeParams& p, int i0, int i1, bool report) {
  const bool ok0 = i0 >= 0 && (int64_t)i0 < p.num_rows;
  const bool ok1 = i1 >= 0 && (int64_t)i1 < p.num_rows;
  const bool bad = (i0 != -1 && !ok0) || (i1 != -1 && !ok1);
  const uint32_t lo = __ballot_sync(0xffffffffu, ok0), hi = __ballot_sync(0xffffffffu, ok1);
  if (report && __any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(p.status, STATUS_INDEX);
  return (uint64_t)lo | ((uint64_t)hi << 32);
}

// The pages of one dense request seen through a 64-tile window: lane i holds
// the page of tile base+i (cur) and base+32+i (nxt); moving the window loads
// the block after next, 32 tiles before it is used.
struct PageWindow {
  int b, base, cur, nxt;
  __device__ __forceinline__ void start(const DecodeParams& p, int b_, int t0) {
    b = b_;
    base = t0;
    cur = load_pages32(p, b, t0);
    nxt = load_pages32(p, b, t0 + 32);
  }
  __device__ __forceinline__ void advance(const DecodeParams& p, int t) {
    while (t - base >= 32) {
      base += 32;
      cur = nxt;
      nxt = load_pages32(p, b, base + 32);
    }
  }
  // t - base in [0, 64); every lane calls it with the same t
  __device__ __forceinline__ int get(int t) const {
    const int d = t - base;
    const int a = __shfl_sync(0xffffffffu, cur, d & 31);
    const int c = __shfl_sync(0xffffffffu, nxt, d & 31);
    return d < 32 ? a : c;
  }
};

// masks of consecutive tiles t0, t0+1, ... of one piece (one call per tile)
template <bool kSparse>
struct MaskStream {
  int v, len;
  PageWindow w;
  // sparse: indices of tiles t, t+1, t+2 (each lane holds entries lane and
  // lane + 32 of a tile). Tile t+3 is fetched by prefetch(), which the caller
  // issues after its work on tile t, so that no index load is outstanding
  // while that work runs.
  int a0, a1, c0, c1, e0, e1;
  __device__ __forceinline__ void start(const DecodeParams& p, const Piece& pc) {
    v = pc.v;
    len = pc.len;
    if constexpr (kSparse) {
      sparse_fetch(p, v, pc.t0, a0, a1);
      sparse_fetch(p, v, pc.t0 + 1, c0, c1);
      sparse_fetch(p, v, pc.t0 + 2, e0, e1);
    } else {
      w.start(p, v % p.batch, pc.t0);
    }
  }
  __device__ __forceinline__ uint64_t next(const DecodeParams& p, int t, bool report) {
    if constexpr (kSparse) {
      return sparse_mask(p, a0, a1, report);
    } else {
      w.advance(p, t);
      return dense_mask(p, w.get(t), t, len, report);
    }
  }
  // after the work on tile t: shift the ring and fetch tile t+3
  __device__ __forceinline__ void prefetch(const DecodeParams& p, int t) {
    if constexpr (kSparse) {
      a0 = c0;
      a1 = c1;
      c0 = e0;
      c1 = e1;
      sparse_fetch(p, v, t + 3, e0, e1);
    }
  }
};

// ---- exact recompute of flagged rows (dense 16-bit caches) ----
// The decode kernel flags a (query position, head) row when the two halves of
// its scores disagree too much for the fp16 factors the pair exchanges; the
// combine recomputes such a row here, from q and the cache rows, with plain
// fp32 arithmetic.
template <bool kF16>
__device__ __forceinline__ float half_to_f32(uint32_t bits16) {
  if constexpr (kF16) return __half2float(__ushort_as_half((unsigned short)bits16));
  else return __uint_as_float(bits16 << 16);
}
// q . K over the 576 dims of 16-bit rows, in fp32 and a fixed order
template <bool kF16>
__device__ __forceinline__ float dot576(const uint16_t* q, const uint16_t* k) {
  const uint4* qa = reinterpret_cast<const uint4*>(q);
  const uint4* ka = reinterpret_cast<const uint4*>(k);
  float acc = 0.f;
#pragma unroll 2
  for (int c = 0; c < kDK / 8; ++c) {
    const uint4 x = __ldg(qa + c), y = __ldg(ka + c);
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc = fmaf(half_to_f32<kF16>(xw[j] & 0xFFFFu), half_to_f32<kF16>(yw[j] & 0xFFFFu), acc);
      acc = fmaf(half_to_f32<kF16>(xw[j] >> 16), half_to_f32<kF16>(yw[j] >> 16), acc);
    }
  }
  return acc;
}

// Attention of head h of query position i of request b over all its visible
// tokens, by the whole block (256 threads): an online softmax over chunks of
// 256 tokens, one exact score per thread, then each thread accumulates two of
// the 512 output dims over the chunk. Pages out of range are skipped, as in
// the decode kernel.
template <typename OutT>
__device__ void exact_head(const CombineParams& p, int b, int i, int h) {
  constexpr bool kF16 = std::is_same<OutT, __half>::value;
  __shared__ float sP[256];
  __shared__ int64_t sRow[256];
  __shared__ float red_m[8], red_s[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = p.seqlens[b];
  if (p.causal) L = L - p.s_q + 1 + i;
  L = L < 0 ? 0 : L;
  const int64_t qv = (int64_t)b * p.s_q + i;
  const uint16_t* qrow = static_cast<const uint16_t*>(p.q) + (qv * p.h_q + h) * kDK;
  const uint16_t* kv = reinterpret_cast<const uint16_t*>(p.kv);
  float m = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f;
  for (int c0 = 0; c0 < L; c0 += 256) {
    const int t = c0 + tid;
    float s = -INFINITY;
    int64_t row = -1;
    if (t < L && t / kTile < p.max_blocks) {
      const int page = __ldg(p.block_table + (int64_t)b * p.max_blocks + t / kTile);
      if (page >= 0 && page < p.num_blocks) {
        row = (int64_t)page * kTile + t % kTile;
        s = dot576<kF16>(qrow, kv + row * kDK) * p.scale_log2;
      }
    }
    float mx = s;
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_m[warp] = mx;
    __syncthreads();
    mx = red_m[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red_m[w]);
    const float m_new = fmaxf(m, mx);
    const float alpha = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
    const float pt = (s == -INFINITY) ? 0.f : exp2f(s - m_new);
    sP[tid] = pt;
    sRow[tid] = row;
    float sm = pt;
#pragma unroll
    for (int o = 16; o; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) red_s[warp] = sm;
    __syncthreads();
    sm = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sm += red_s[w];
    l = l * alpha + sm;
    o0 *= alpha;
    o1 *= alpha;
    const int n = L - c0 < 256 ? L - c0 : 256;
    for (int j = 0; j < n; ++j) {
      const float pj = sP[j];
      if (pj != 0.f) {
        const uint16_t* vr = kv + sRow[j] * kDK;
        o0 = fmaf(pj, half_to_f32<kF16>(vr[tid]), o0);
        o1 = fmaf(pj, half_to_f32<kF16>(vr[tid + 256]), o1);
      }
    }
    m = m_new;
    __syncthreads();
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  OutT* orow = reinterpret_cast<OutT*>(p.out) + (qv * p.h_q + h) * kDV;
  if constexpr (kF16) {
    orow[tid] = __float2half_rn(o0 * inv);
    orow[tid + 256] = __float2half_rn(o1 * inv);
  } else {
    orow[tid] = __float2bfloat16_rn(o0 * inv);
    orow[tid + 256] = __float2bfloat16_rn(o1 * inv);
  }
  if (tid == 0) p.lse[qv * p.h_q + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

// Merge the split partials of each virtual request. grid = (vreq, h_q/16),
// block = 256: 16 heads per block, each thread 32 of one head's 512 dims.
// Requests with a single piece were finished by the decode kernel; requests
// with no visible token get out = 0, lse = -inf here.
// kNu: units of 8 dims per thread, 8 / gridDim.z (8 with one block per 16
// heads, 1 when eight blocks share them).
template <typename OutT, int kNu>
__global__ void __launch_bounds__(256) mla_combine_kernel(CombineParams p) {
  pdl_launch_dependents();  // a following schedule kernel may launch; it waits for this grid
  pdl_wait();  // the decode grid has completed and its writes are visible
  const int v = blockIdx.x;
  const int b = v % p.batch, i = v / p.batch;
  // the request's split range and its flag word are loaded together
  const int off = p.split_off[v];
  const int ns = p.split_off[v + 1] - off;
  // rows the decode kernel flagged (bit k: head 16*blockIdx.y + k) are
  // recomputed exactly and left out of the merge below; their bits are cleared
  uint32_t fmask = 0u;
  if (p.exact_flags) {
    const int h0 = blockIdx.y * 16;
    uint32_t* fw = p.exact_flags + (int64_t)v * 4 + (h0 >> 5);
    fmask = (*fw >> (h0 & 31)) & 0xFFFFu;
    if (fmask) {
      for (int k = 0; k < 16; ++k)
        if ((fmask >> k) & 1u) exact_head<OutT>(p, b, i, h0 + k);
      if (threadIdx.x == 0) atomicAnd(fw, ~(0xFFFFu << (h0 & 31)));
    }
  }
  if (ns == 1) return;
  // Thread t merges, for head 16*blockIdx.y + hl, four dims (4*half ..
  // 4*half+3) of each of kNu units of 8 dims, units u0 .. u0+kNu-1. The 32
  // threads of a warp then read one unit of 16 heads, 512 contiguous bytes of
  // the o_part layout (opart_index). gridDim.z blocks share a request's 64
  // units (more blocks when there are few heads; 1 whenever rows may be
  // flagged for the exact recompute above, which each block would redo).
  const int t = threadIdx.x;
  const int hl = (t >> 1) & 15, half = t & 1, ug = t >> 5;
  const int u0 = (8 * (int)blockIdx.z + ug) * kNu;
  const int h = blockIdx.y * 16 + hl;
  if (h >= p.h_q || ((fmask >> hl) & 1u)) return;  // recomputed above
  const int64_t row = ((int64_t)(b * p.s_q + i) * p.h_q + h);
  OutT* orow = reinterpret_cast<OutT*>(p.out) + row * kDV;
  const int64_t ustride = (int64_t)p.h_q * 8;  // floats from one unit to the next
  const int64_t sstride = 64 * ustride;        // and from one split to the next
  const float* src = p.o_part + opart_index(off, p.h_q, h, 8 * u0) + 4 * half;
  const float* lsp = p.lse_part + (int64_t)off * p.h_q + h;
  // The first kPre pieces' partials (16 units in all: two pieces of 8 units,
  // or sixteen of one) are loaded together with every piece's lse, so that a
  // request cut into up to kPre pieces costs one round trip to memory.
  constexpr int kPre = 16 / kNu;
  float4 x[kPre][kNu];
  float ls[kPre];
  float mx = -INFINITY;
#pragma unroll
  for (int s = 0; s < kPre; ++s) {
    ls[s] = -INFINITY;
    if (s < ns) {
#pragma unroll
      for (int k = 0; k < kNu; ++k) x[s][k] = *reinterpret_cast<const float4*>(src + s * sstride + k * ustride);
      ls[s] = lsp[(int64_t)s * p.h_q];
    }
  }
#pragma unroll
  for (int s = 0; s < kPre; ++s) mx = fmaxf(mx, ls[s]);
  for (int s = kPre; s < ns; ++s) mx = fmaxf(mx, lsp[(int64_t)s * p.h_q]);
  float4 acc[kNu];
#pragma unroll
  for (int k = 0; k < kNu; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  // o += e^{lse_s - m} o_s, in the order of the pieces
  auto add = [&](const float4(&xs)[kNu], float l_s) {
    if (l_s == -INFINITY) return;  // an empty piece, or none (m is finite otherwise)
    const float w = expf(l_s - mx);
    wsum += w;
#pragma unroll
    for (int k = 0; k < kNu; ++k) {
      acc[k].x += w * xs[k].x;
      acc[k].y += w * xs[k].y;
      acc[k].z += w * xs[k].z;
      acc[k].w += w * xs[k].w;
    }
  };
#pragma unroll
  for (int s = 0; s < kPre; ++s) add(x[s], ls[s]);
  for (int s = kPre; s < ns; ++s) {
    float4 xs[kNu];
#pragma unroll
    for (int k = 0; k < kNu; ++k) xs[k] = *reinterpret_cast<const float4*>(src + s * sstride + k * ustride);
    add(xs, lsp[(int64_t)s * p.h_q]);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int k = 0; k < kNu; ++k) {
    const int d = 8 * (u0 + k) + 4 * half;
    uint32_t lo, hi;
    if constexpr (std::is_same<OutT, __half>::value) {
      lo = pack_f16x2(acc[k].x * inv, acc[k].y * inv);
      hi = pack_f16x2(acc[k].z * inv, acc[k].w * inv);
    } else {
      lo = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
      hi = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
    }
    *reinterpret_cast<uint2*>(orow + d) = make_uint2(lo, hi);
  }
  if (u0 == 0 && half == 0) p.lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

}  // namespace mla
