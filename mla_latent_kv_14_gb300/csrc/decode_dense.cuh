// decode_dense.cuh -- MLA decode, 128 heads, over a latent cache of 16-bit,
// 656-byte FP8 or V4.1 (528-byte FP8, 288-byte FP4) rows, read through a block
// table or an index list, sm_103a.
//
// What one 2-CTA cluster computes. A persistent cluster owns one range of the
// split-KV schedule (a list of (virtual request, tile range) pieces). For a
// piece it keeps, for all 128 heads, the online-softmax state (m, l) and the
// 512-wide latent output O, and walks the piece's 64-token tiles:
//   S  = Q K^T              (128 heads x 64 tokens, contraction over 576, or
//                            512 for the V4.1 rows)
//   P  = exp(S*scale - m)   (online softmax with running max / sum)
//   O += P V                (V = the first 512 dims of the same rows)
// ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §五 flashDecode, §六 absorbed MQA
// shape, §七 split-KV; "FlashMLA 实战", §最小调用).
//
// How the work is laid out on GB300. The fp32 O for 128 heads x 512 fills the
// whole 128-lane x 512-column tensor memory of one SM, so the two CTAs of the
// cluster split the latent dimension: CTA r keeps O[:, 256r : 256r+256] in TMEM
// (256 columns) and loads only its own part of Q and of every KV tile: CTA r
// the latent dims [256r, 256r+256) and the RoPE dims [512+32r, 544+32r).
// Each CTA computes a partial score S_r over its dims with single-CTA UMMA
// (M=128 heads, N=64 tokens). Instead of exchanging S_r, each CTA exponentiates
// it, E_r = exp2((S_r - m_r) * scale*log2e + 15) with m_r its partial row max,
// and sends E_r as fp16 plus m_r: exp(S_0 + S_1 - m) = E_0 * E_1 *
// exp(m_0 + m_1 - m) * 2^-30 is exact algebra, so both CTAs form the same P
// from identical fp16 operands (commutative products) and accumulate P . V
// for their own half of the latent (M=128, N=256, K=64). The 2^15 shift puts
// 28 binades below each half's maximum in fp16's normal range, and its
// subnormals keep an absolute precision of 2^-25 below that, so each product
// is known to a relative 2^-10 or an absolute 2^-10 (of 2^30). A row whose
// products sum to at least 2^8 is therefore certified to within 2^-12; that
// fails only when the two halves' scores disagree by more than about 22
// binades. Such a row is flagged and the combine kernel recomputes it exactly
// (16-bit caches) or it is reported as out of range (quantised rows). No tensor-core work is
// duplicated and no KV byte is read twice; the exchange is 16.5 KB per tile
// and direction. (Prior art on the pages: the Hopper kernel splits O between
// two warpgroups -- seesaw -- because the register file is full, and the FP8
// kernel pairs two CTAs over DSM -- Crossover; here the pair exists because
// TMEM is full.)
//
// Memory map. TMEM (512 columns): the O half [0,256); S, one buffer
// [256,320); P of tiles g&1 = 0, 1 at [320,352) and [352,384), 16-bit pairs,
// read by P . V as its A operand straight from TMEM; and this CTA's 256 latent
// dims of Q as the A operand of QK^T [384,512) (column j = the 16-bit pair
// (2j, 2j+1) of head row = lane). Shared memory: the peer's message (E_r fp16
// 128x64 + m_r + the tile mask, 16.5 KB), this CTA's own message staged for
// the copy, the CTA's 32 RoPE dims of Q (8 KB) and a ring of KV tiles (36 KB
// each: four 64-wide latent chunks, 128-byte swizzled, loaded as one 3-D TMA
// box, and one 32-wide RoPE chunk, 64-byte swizzled): 5 slots for 16-bit
// caches; 3 for quantised rows (32 KB without the RoPE chunk for the V4.1
// rows), whose raw codes, scales and (656-byte rows) RoPE dims stage in 3 more
// slots (dense: TMA; sparse: TMA gather4, four rows per copy); the dequant
// warps fill the operand slot from them.
//
// Warp roles. Warp 0: producer (TMA; the whole warp in the sparse mode).
// Warp 1: owns TMEM; lane 0 issues QK^T. Warp kPvWarp (2, or 14 for quantised
// rows): lane 0 issues P . V, so a P . V never waits behind the issue of a
// QK^T tile; it holds a ready P . V back while a QK^T is executing, so that
// it fills the pipe while the E warps read S instead of delaying S. Warps 2-3
// and 12-13 (quantised rows): codes x scale -> fp16 operand tiles. Warps 4-7 (E):
// read S, form E_r and the row max, stage them and send them to the peer with
// one bulk shared-to-shared copy; they also copy each piece's Q rows into
// TMEM. Warps 8-11 (P): receive the peer's message, form P into TMEM, rescale
// O when the running max moves by more than 2^8, and write the piece's
// output. Warp w of the E and P groups serves TMEM lanes (heads) 32*(w%4) ..
// +31.
//
// Pipeline. Every hand-off is an mbarrier; every wait is bounded (a wait that
// gives up sets a status bit and the kernel unwinds). Measured on GB300 with
// per-tile clock stamps: the tile period (about 2,150 cycles for 16-bit
// caches) is set by two loops of about that length -- QK^T issue and
// completion plus the E warps' read of the single S buffer, and the exchange
// buffers (a 16.5 KB copy between the SMs of a pair lands about 1,250 cycles
// after it is issued) -- with the ring deep enough to cover the rest. A
// single-CTA UMMA with N=64 costs as much as one with N=128 (about 64 cycles
// at M=128, K=16), so QK^T of a tile takes about 1,150 cycles of the tensor
// pipe and P . V about 512.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "params.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace mla {
namespace dense {

// 16-bit caches (576-wide rows); 656-byte FP8 rows; the V4.1 rows of 512
// values: 528-byte FP8 (e4m3 + UE8M0 per 32) and 288-byte FP4 (e2m1 + e4m3
// per 16); each quantised row format paged (dense) or token-sparse
enum : int {
  MODE_BF16 = 0, MODE_FP16 = 1, MODE_FP8 = 2, MODE_FP8_SPARSE = 3,
  MODE_V41_FP8 = 4, MODE_V41_FP8_SPARSE = 5, MODE_V41_FP4 = 6, MODE_V41_FP4_SPARSE = 7
};

constexpr int kKChunk = 64 * 128;          // 64 tokens x 64 x 2 B
constexpr int kRChunk = 64 * 64;           // 64 tokens x 32 RoPE dims x 2 B
constexpr int kSlot = 4 * kKChunk + kRChunk;
constexpr int kThreads = 384;              // 16-bit caches (quantised rows: Cfg::kThreads)
constexpr int kEWarps = 4;                 // warps 4-7: exponentiate and send
constexpr int kPWarps = 4;                 // warps 8-11: receive, form P, epilogue
constexpr int kDequantWarps = 4;           // warps 2-3 and 12-13 (quantised rows)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;            // S at columns 256..319 (one buffer)
constexpr uint32_t kColP = 320;            // P of tile g: 16-bit pairs at columns 320 + 32*(g&1)
constexpr uint32_t kColQ = 384;            // Q latent (bf16 pairs) at columns 384..511
constexpr uint32_t kXE = 128 * 128;                     // E_r: 128 rows x 64 fp16
constexpr uint32_t kXM = kXE;                           // + m_r per row (fp32)
constexpr uint32_t kXMask = kXM + 128 * 4;              // + validity mask of the tile (64 bits)
constexpr uint32_t kXBytes = kXMask + 16;
// E_r = 2^(s_r - m_r + kEShift): fp16's normal range then holds every token
// within 28 binades of the half's own maximum (2^-13 .. 2^15), and below that
// its subnormals keep an absolute precision of 2^-25
constexpr float kEShift = 15.0f;
// A row of a tile is certified when the sum of its products E_own E_peer is at
// least kCertify: every product is then known to a relative 2^-10 or an
// absolute 2^-10, so the 64 tokens' absolute errors add up to at most 2^-12 of
// the sum (about 22 binades of disagreement between the two halves)
constexpr float kCertify = 256.0f;
constexpr uint32_t kXStride = 17 * 1024;
constexpr uint32_t kEBar = 1;                           // named barrier of the 128 E-warp threads
// FP8 rows (656 B): e4m3 [0,512), 4 fp32 scales [512,528), 64 bf16 RoPE [528,656)
// V4.1 FP8 rows (528 B): e4m3 [0,512), 16 UE8M0 scales [512,528)
// V4.1 FP4 rows (288 B): e2m1 [0,256) (value 2i in the low nibble of byte i),
// 32 e4m3 scales [256,288)

#ifndef V41_FP4_NS
#define V41_FP4_NS 3
#endif
#ifndef V41_FP8_NS
#define V41_FP8_NS 3
#endif
// per-mode layout (offsets from a 1024-B aligned base) and barrier indices
template <int kMode>
struct Cfg {
  static constexpr bool kFp16 = kMode == MODE_FP16;
  static constexpr bool kQuant = kMode >= MODE_FP8;        // quantised rows: dequant warps
  static constexpr bool kV41 = kMode >= MODE_V41_FP8;      // 512-value rows, no separate RoPE part
  static constexpr bool kFp4 = kMode >= MODE_V41_FP4;
  static constexpr bool kSparse = kMode == MODE_FP8_SPARSE || kMode == MODE_V41_FP8_SPARSE ||
                                  kMode == MODE_V41_FP4_SPARSE;
  // 16-bit operand type of the latent QK^T and P . V: bf16 for bf16 caches;
  // fp16 for fp16 caches and for every quantised row, whose products are
  // formed in fp16 (cheaper to form than bf16, and exact in the ranges below)
  static constexpr bool kLatBf16 = !(kFp16 || kQuant);
  // operand slot: four 64-wide chunks and, unless the row is a V4.1 row, a
  // 32-wide RoPE chunk
  static constexpr uint32_t kSlotBytes = kV41 ? 4 * kKChunk : kSlot;
  static constexpr int kNS = kQuant ? (kFp4 ? V41_FP4_NS : (kV41 ? V41_FP8_NS : 3)) : 5;  // KV ring slots (tiles)
  // quantised rows: two more dequant warps (12, 13) and the P . V issuer (14)
  static constexpr int kThreads = kQuant ? 480 : 384;
  static constexpr int kPvWarp = kQuant ? 14 : 2;         // its lane 0 issues P . V
  static constexpr int kRawNS = 3;                        // raw staging slots
  static constexpr uint32_t kRowBytes = kFp4 ? 288 : (kV41 ? 528 : 656);
  static constexpr uint32_t kRawRow = kFp4 ? 128 : 256;   // this CTA's data bytes of a row
  static constexpr uint32_t kRawLat = 64 * kRawRow;
  // 16 scale bytes per row (656: the 4 fp32 scales; 528: the 16 UE8M0 scales;
  // 288: this CTA's 16 e4m3 scales); the sparse gather writes them four rows
  // (64 B) at a time into 128-B aligned units
  static constexpr uint32_t kRawSc = kSparse ? 16 * 128 : 64 * 16;
  // 656-byte rows: this CTA's 32 RoPE dims (bf16) of the 64 rows, 64-byte
  // swizzled like the operand slot's RoPE chunk (both 512-B aligned), copied
  // there by the dequant warps; so the producer never waits for a free operand
  // slot and its raw loads run kRawNS tiles ahead
  static constexpr uint32_t kRawRope = kV41 ? 0 : kRChunk;
  static constexpr uint32_t kRawSlot = kRawLat + kRawSc + kRawRope;
  static constexpr uint32_t OFF_XR = 0;                  // peer's message
  static constexpr uint32_t OFF_XS = OFF_XR + kXStride;  // own message, staged for the copy
  static constexpr uint32_t OFF_QR = OFF_XS + kXStride;  // 32 RoPE dims of Q: 128 rows x 64 B
  static constexpr uint32_t OFF_RING = OFF_QR + (kV41 ? 0 : 128 * 64);
  static constexpr uint32_t OFF_RAW = OFF_RING + kNS * kSlotBytes;
  static constexpr uint32_t OFF_BAR = OFF_RAW + (kQuant ? kRawNS * kRawSlot : 0);
  static constexpr uint32_t B_FULL = 0, B_EMPTY = B_FULL + kNS, B_QFULL = B_EMPTY + kNS, B_QEMPTY = B_QFULL + 1,
                            B_SFULL = B_QEMPTY + 1, B_SEMPTY = B_SFULL + 1, B_PFULL = B_SEMPTY + 1,
                            B_PEMPTY = B_PFULL + 2, B_OEMPTY = B_PEMPTY + 2, B_XFULL = B_OEMPTY + 1,
                            B_XEMPTY = B_XFULL + 1, B_DRAIN = B_XEMPTY + 1, B_XSFREE = B_DRAIN + 1,
                            B_XSFULL = B_XSFREE + 1, B_RFULL = B_XSFULL + 1,
                            B_REMPTY = B_RFULL + kRawNS, B_DRAIN2 = B_REMPTY + kRawNS,
                            B_STALL = B_DRAIN2 + 1, B_COUNT = B_STALL + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 8 * B_COUNT;   // tmem slot, abort flag, ok flag
  static constexpr uint32_t kSmemBytes = OFF_MISC + 64 + 1024;  // + alignment slack
};
static_assert(Cfg<MODE_BF16>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_FP8_SPARSE>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_FP8>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_V41_FP8>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_V41_FP8_SPARSE>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_V41_FP4>::kSmemBytes <= 232448, "shared memory");
static_assert(Cfg<MODE_V41_FP4_SPARSE>::kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ bool warp_ok(bool x) { return __all_sync(0xffffffffu, x); }

// The reference max of the online softmax, moved lazily: the running max m
// moves to the tile's row max Mt only when Mt exceeds it by more than 2^8, so
// that P = 2^(s - m_use) <= 256 and O is rescaled rarely.
struct RowRef {
  float m_use, alpha;
  bool resc, live;
  __device__ __forceinline__ RowRef(float m, float Mt) {
    const float m_new = fmaxf(m, Mt);
    resc = m_new > m + 8.0f;
    m_use = resc ? m_new : m;
    alpha = resc ? exp2_approx(m - m_new) : 1.0f;
    live = Mt != -INFINITY;
  }
};

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// 2^k as an fp16 pair: normal for k in [-14, 15], subnormal down to 2^-24,
// zero below (k above 15 does not occur: such blocks are reported)
__device__ __forceinline__ uint32_t f16x2_pow2(int k) {
  const uint32_t h = k >= -14 ? (uint32_t)(k + 15) << 10 : (k >= -24 ? 1u << (k + 24) : 0u);
  return h | (h << 16);
}
// four bytes of e2m1 pairs -> four f16 pairs (exact); byte i gives h[i], its
// low nibble in the low half
__device__ __forceinline__ void cvt_e2m1x4_f16x2(uint32_t w, uint32_t* h) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}


template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kMode>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_qr, const __grid_constant__ CUtensorMap tm_kv,
                      const __grid_constant__ CUtensorMap tm_kvr, const __grid_constant__ CUtensorMap tm_sc,
                      const DecodeParams p) {
  using C = Cfg<kMode>;
  constexpr bool kFp16 = C::kFp16, kQuant = C::kQuant, kV41 = C::kV41, kFp4 = C::kFp4,
                 kSparse = C::kSparse;
  constexpr int NS = C::kNS;
  using OutT = typename std::conditional<kFp16, __half, __nv_bfloat16>::type;
  constexpr int kDQ = kV41 ? 512 : kDK;  // query row width
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int part = (int)cluster_id_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  auto bar = [&](uint32_t i) { return sb + C::OFF_BAR + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* tmem_slot = misc + 0;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* ok_flag = misc + 2;
  volatile uint32_t* qk_started = misc + 3;  // QK^T tiles whose issue has begun
  const Guard guard{abort_flag, p.status, kWaitLimitCycles};

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      // the producer's copy (16-bit caches) or the dequant warps (quantised rows)
      mbar_init(bar(C::B_FULL + s), kQuant ? kDequantWarps : 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_QFULL), kEWarps + 1);  // E warps (latent into TMEM) + producer (RoPE TMA)
    mbar_init(bar(C::B_QEMPTY), 1);
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_SEMPTY), kEWarps);
    mbar_init(bar(C::B_XSFREE), kPWarps);  // P warps have read XS
    mbar_init(bar(C::B_XSFULL), 1);        // E warps have staged XS
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_PFULL + s), kPWarps);  // P of tile g (g&1 = s) is in TMEM
      mbar_init(bar(C::B_PEMPTY + s), 1);       // its P . V is done
    }
    mbar_init(bar(C::B_OEMPTY), kPWarps);
    mbar_init(bar(C::B_XFULL), 1);              // own expect_tx + the peer's copied bytes
    mbar_init(bar(C::B_XEMPTY), kPWarps);  // one arrive per peer P warp
    mbar_init(bar(C::B_DRAIN), 1);
    mbar_init(bar(C::B_DRAIN2), 1);
    mbar_init(bar(C::B_STALL), 1);
    for (int s = 0; s < C::kRawNS; ++s) {
      mbar_init(bar(C::B_RFULL + s), 1);
      mbar_init(bar(C::B_REMPTY + s), kDequantWarps);
    }
    *abort_flag = 0u;
    *qk_started = 0u;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote access
  tc_fence_after();
  // Everything above reads no global memory. The schedule, and possibly the
  // query, cache and tables, come from kernels earlier on the stream; the
  // launch is a programmatic dependent launch, so wait for them here. The
  // metadata header is loaded before the lengths are hashed, so that both
  // reads are in flight together.
  pdl_wait();
  int32_t hdr[H_WORDS];
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < H_WORDS; ++k) hdr[k] = p.meta[k];
  }
  const uint32_t fp = warp == 0 ? lengths_hash_warp(p.seqlens, p.batch, p.topk) : 0u;
  if (threadIdx.x == 0) {
    *ok_flag = header_matches(hdr, p, kTile, fp) ? 1u : 0u;
    if (!*ok_flag && rank == 0) atomicOr(p.status, STATUS_STALE);
    if (*ok_flag && p.stall_cycles) {
      // test hook: a bounded wait on a barrier nothing arrives at gives up
      // and reports STATUS_TIMEOUT; nothing has been issued yet, so the CTA
      // simply skips its work
      const Guard g_stall{abort_flag, p.status, p.stall_cycles};
      if (!wait(bar(C::B_STALL), 0, g_stall)) *ok_flag = 0u;
    }
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  const bool ok = *ok_flag != 0u;

  if (ok && warp == 0 && (kSparse || lane == 0)) {
    // ---------------- producer: RoPE dims of Q per piece, KV per tile ----------------
    if (lane == 0) {
      prefetch_tmap(&tm_kv);
      if constexpr (!kV41) {
        prefetch_tmap(&tm_qr);
        prefetch_tmap(&tm_kvr);
      }
      if constexpr (kQuant) prefetch_tmap(&tm_sc);
    }
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_last();
    const int xr = 512 + 32 * (int)rank;  // RoPE column of this CTA (bf16 caches)
    // byte column of the scales this CTA reads (288-byte rows: its own 16)
    const int kScX = kFp4 ? 256 + 16 * (int)rank : 512;
    PieceIter it(p, part);
    Piece pc;
    int g = 0, qn = 0;
    int last_g[NS];
    for (int s = 0; s < NS; ++s) last_g[s] = -1;
    int last_rg[C::kRawNS];
    for (int s = 0; s < C::kRawNS; ++s) last_rg[s] = -1;
    int q_last = -1;
    bool stop = false;
    // block-table entries are loaded one iteration before they are used
    auto raw_page = [&](int b, int t) {
      return t < p.max_blocks ? __ldg(p.block_table + (int64_t)b * p.max_blocks + t) : -1;
    };
    auto sane = [&](int page) { return (page < 0 || page >= p.num_blocks) ? 0 : page; };  // bad pages are masked
    while (!stop && it.next(pc)) {
      const int b = pc.v % p.batch, i = pc.v / p.batch;
      if (lane == 0) {
        if (!wait(bar(C::B_QEMPTY), (qn & 1) ^ 1, guard)) stop = true;
        else if constexpr (kV41) {
          mbar_arrive(bar(C::B_QFULL));  // no RoPE part: the E warps load all of Q
        } else {
          mbar_arrive_expect_tx(bar(C::B_QFULL), 128 * 64);
          tma_load_2d(sb + C::OFF_QR, &tm_qr, bar(C::B_QFULL), xr, (b * p.s_q + i) * 128, pol_q);
          q_last = qn;
        }
      }
      if (kSparse && !warp_ok(!stop)) stop = true;
      if (stop) break;
      ++qn;
      int pg_next = 0;               // dense: page of tile t, loaded one tile ahead
      // sparse: indices of tiles t, t+1, t+2, loaded three tiles ahead, so that
      // the gathers of tile t find its indices in registers
      int n0 = 0, n1 = 0, m0 = 0, m1 = 0, k0 = 0, k1 = 0;
      if constexpr (!kSparse) {
        pg_next = raw_page(b, pc.t0);
      } else {
        sparse_fetch(p, pc.v, pc.t0, n0, n1);
        sparse_fetch(p, pc.v, pc.t0 + 1, m0, m1);
        sparse_fetch(p, pc.v, pc.t0 + 2, k0, k1);
      }
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        const int s = g % NS;
        if constexpr (!kSparse) {
          const int page = sane(pg_next);
          pg_next = raw_page(b, t + 1);
          if constexpr (kQuant) {
            // raw codes + scales into the staging ring, converted by the dequant warps
            const int rs = g % C::kRawNS;
            if (!wait(bar(C::B_REMPTY + rs), ((g / C::kRawNS) & 1) ^ 1, guard)) { stop = true; break; }
            const uint32_t raw = sb + C::OFF_RAW + rs * C::kRawSlot;
            mbar_arrive_expect_tx(bar(C::B_RFULL + rs), C::kRawSlot);
            tma_load_2d(raw, &tm_kv, bar(C::B_RFULL + rs), (int)C::kRawRow * (int)rank, page * kTile, pol_kv);
            tma_load_2d(raw + C::kRawLat, &tm_sc, bar(C::B_RFULL + rs), kScX, page * kTile, pol_kv);
            if constexpr (!kV41)  // the RoPE dims are bf16 in the row
              tma_load_2d(raw + C::kRawLat + C::kRawSc, &tm_kvr, bar(C::B_RFULL + rs), 528 + 64 * (int)rank,
                          page * kTile, pol_kv);
            last_rg[rs] = g;
            continue;  // the dequant warps fill the operand slot
          }
          if (!wait(bar(C::B_EMPTY + s), ((g / NS) & 1) ^ 1, guard)) { stop = true; break; }
          const uint32_t slot = sb + C::OFF_RING + s * C::kSlotBytes;
          mbar_arrive_expect_tx(bar(C::B_FULL + s), kSlot);
          tma_load_3d(slot, &tm_kv, bar(C::B_FULL + s), 0, page * kTile, 4 * (int)rank, pol_kv);
          tma_load_2d(slot + 4 * kKChunk, &tm_kvr, bar(C::B_FULL + s), xr, page * kTile, pol_kv);
          last_g[s] = g;
        } else {
          // sparse: TMA gather4, four rows per copy; lane j < 16 fetches rows
          // 4j .. 4j+3 of the tile for each field (this CTA's data bytes, the
          // 16 scale bytes, and for 656-byte rows its 64 RoPE bytes). A row
          // that is -1 or out of range is fetched as row 0 and masked later.
          const int rs = g % C::kRawNS;
          const int idx[2] = {n0, n1};
          n0 = m0;
          n1 = m1;
          m0 = k0;
          m1 = k1;
          if (t + 3 < pc.t1) sparse_fetch(p, pc.v, t + 3, k0, k1);  // consumed three tiles on
          if (!warp_ok(wait(bar(C::B_REMPTY + rs), ((g / C::kRawNS) & 1) ^ 1, guard))) { stop = true; break; }
          const uint32_t raw = sb + C::OFF_RAW + rs * C::kRawSlot;
          const int s0 = (idx[0] >= 0 && (int64_t)idx[0] < p.num_rows) ? idx[0] : 0;
          const int s1 = (idx[1] >= 0 && (int64_t)idx[1] < p.num_rows) ? idx[1] : 0;
          int r[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int row = 4 * (lane & 15) + q;
            const int a = __shfl_sync(0xffffffffu, s0, row & 31);
            const int c = __shfl_sync(0xffffffffu, s1, row & 31);
            r[q] = row < 32 ? a : c;
          }
          if (lane == 0) mbar_arrive_expect_tx(bar(C::B_RFULL + rs), 64u * (C::kRawRow + 16) + C::kRawRope);
          __syncwarp();
          if (lane < 16) {
            const uint32_t fb = bar(C::B_RFULL + rs);
            tma_gather4(raw + lane * 4 * C::kRawRow, &tm_kv, fb, (int)C::kRawRow * (int)rank, r[0], r[1], r[2], r[3],
                        pol_kv);
            tma_gather4(raw + C::kRawLat + lane * 128, &tm_sc, fb, kScX, r[0], r[1], r[2], r[3], pol_kv);
            // 656-byte rows: the RoPE dims (bf16), 64-byte swizzled by the copy
            if constexpr (!kV41)
              tma_gather4(raw + C::kRawLat + C::kRawSc + lane * 4 * 64, &tm_kvr, fb, 528 + 64 * (int)rank, r[0], r[1],
                          r[2], r[3], pol_kv);
          }
          last_rg[rs] = g;
        }
      }
    }
    // never leave with a copy in flight into this CTA's shared memory
    if (lane == 0) {
      for (int s = 0; s < NS; ++s)
        if (last_g[s] >= 0) {
          const uint64_t t_0 = cycles();
          while (!mbar_try_wait(bar(C::B_FULL + s), (last_g[s] / NS) & 1) && cycles() - t_0 < kDrainLimitCycles) {}
        }
      for (int s = 0; s < C::kRawNS; ++s)
        if (last_rg[s] >= 0) {
          const uint64_t t_0 = cycles();
          while (!mbar_try_wait(bar(C::B_RFULL + s), (last_rg[s] / C::kRawNS) & 1) && cycles() - t_0 < kDrainLimitCycles) {}
        }
      if (q_last >= 0) {
        const uint64_t t_0 = cycles();
        while (!mbar_try_wait(bar(C::B_QFULL), q_last & 1) && cycles() - t_0 < kDrainLimitCycles) {}
      }
    }
  } else if (kQuant && ok && (warp == 2 || warp == 3 || warp == 12 || warp == 13)) {
    // ---------------- dequant: codes x block scale -> fp16 operand tiles ----------------
    // (fp16 keeps 11 bits of the product; the latent QK^T and P . V of
    // quantised rows run as fp16 x fp16, the RoPE QK^T of 656-byte rows stays
    // bf16 x bf16). 656: e4m3 x fp32 scale, rounded through the fp16 copy of
    // the scale. 528: e4m3 x 2^k, exact for k in [-15, 7]. 288: e2m1 x e4m3,
    // always exact (magnitudes in [2^-10, 2688]).
    const int tid = (warp < 4 ? warp - 2 : warp - 10) * 32 + lane;  // 0..127 over the four warps
    PieceIter it(p, part);
    Piece pc;
    int g = 0;
    bool failed = false;
    // 656: largest block scale seen: a scale of at most 146 (block amax <=
    // 65408) keeps its fp16 copy at most 146 (an fp16 value), so no product
    // code x scale (|code| <= 448) exceeds fp16's 65504
    float sc_max = 0.f;
    // 528: largest UE8M0 byte seen: up to 134 (k <= 7, block amax <= 448 * 2^7)
    // no product code x 2^k exceeds fp16's 65504
    uint32_t ue_max = 0u;
    while (!failed && it.next(pc)) {
      MaskStream<kSparse> ms;
      ms.start(p, pc);
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        const int rs = g % C::kRawNS, s = g % NS;
        const uint64_t vmask = ms.next(p, t, false);
        if (!warp_ok(wait(bar(C::B_RFULL + rs), (g / C::kRawNS) & 1, guard)) ||
            !warp_ok(wait(bar(C::B_EMPTY + s), ((g / NS) & 1) ^ 1, guard))) {
          failed = true;
          break;
        }
        const uint32_t raw = sb + C::OFF_RAW + rs * C::kRawSlot;
        const uint32_t slot = sb + C::OFF_RING + s * C::kSlotBytes;
        const uint32_t scales = raw + C::kRawLat;
        // The thread converts unit `lane` (8 values) of rows wq, wq + 4, ...,
        // wq + 60; consecutive lanes take consecutive units of one row
        // (conflict-free loads, 16-B swizzled stores). All 16 rows' codes and
        // scales are loaded first and converted after: the shared-memory
        // accesses are ordered asm, so interleaving them row by row would
        // serialise every row's load -> convert -> store chain.
        const int wq = tid >> 5;
        uint32_t r0[16], r1[16], sc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int row = 4 * k + wq;
          // the row's 16 scale bytes: dense 16 B per row; sparse: rows
          // 4k..4k+3 share a 128-B unit
          const uint32_t sc_row = scales + (kSparse ? (row >> 2) * 128 + (row & 3) * 16 : row * 16);
          if constexpr (kFp4) {
            r0[k] = ld_shared_u32(raw + row * 128 + lane * 4);
            sc[k] = ld_shared_u8(sc_row + (lane >> 1));
          } else {
            ld_shared_v2(raw + row * 256 + lane * 8, r0[k], r1[k]);
            sc[k] = kV41 ? ld_shared_u8(sc_row + 8 * rank + (lane >> 2))
                         : ld_shared_u32(sc_row + 4 * (2 * rank + (lane >> 4)));
          }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int row = 4 * k + wq;
          const bool live = (vmask >> row) & 1ull;
          uint32_t w0, w1, w2, w3;
          if constexpr (kFp4) {
            // 8 e2m1 values (4 bytes) x this CTA's e4m3 scale of their 16:
            // both -> f16 exactly, and the product (at most 5 significant
            // bits, magnitude in [2^-10, 2688]) is exact in fp16
            const uint32_t s2 = cvt_e4m3x2_f16x2((uint16_t)(sc[k] | (sc[k] << 8)));
            uint32_t h[4];
            cvt_e2m1x4_f16x2(r0[k], h);
            w0 = mul_f16x2(h[0], s2);
            w1 = mul_f16x2(h[1], s2);
            w2 = mul_f16x2(h[2], s2);
            w3 = mul_f16x2(h[3], s2);
          } else if constexpr (kV41) {
            // 8 e4m3 x 2^k (UE8M0 byte k + 127 of their 32 values): e4m3 ->
            // f16 is exact, and so is the product for k in [-15, 7]; below
            // that it rounds to fp16's subnormal grid (absolute error at most
            // 2^-25)
            const uint32_t ue = sc[k];
            if (live) ue_max = ue > ue_max ? ue : ue_max;
            const uint32_t f2 = f16x2_pow2((int)ue - 127);
            w0 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r0[k] & 0xFFFF)), f2);
            w1 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r0[k] >> 16)), f2);
            w2 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r1[k] & 0xFFFF)), f2);
            w3 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r1[k] >> 16)), f2);
          } else {
            const float scf = __uint_as_float(sc[k]);
            if (live) sc_max = fmaxf(sc_max, scf);
            // e4m3 -> f16 is exact; the product rounds once more through the
            // fp16 copy of the scale (both roundings are below 2^-11 relative)
            const uint32_t sc2 = pack_f16x2(scf, scf);
            w0 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r0[k] & 0xFFFF)), sc2);
            w1 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r0[k] >> 16)), sc2);
            w2 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r1[k] & 0xFFFF)), sc2);
            w3 = mul_f16x2(cvt_e4m3x2_f16x2((uint16_t)(r1[k] >> 16)), sc2);
          }
          if (!live) w0 = w1 = w2 = w3 = 0u;  // masked rows: zero values, whatever the bytes
          st_shared_v4(slot + (lane >> 3) * kKChunk + row * 128 + (((lane & 7) ^ (row & 7)) << 4), w0, w1, w2, w3);
        }
        if constexpr (C::kRawRope > 0) {
          // the RoPE chunk, already in the operand layout (masked tokens'
          // scores are -inf, and RoPE dims are not part of the value)
#pragma unroll
          for (int i = 0; i < (int)(C::kRawRope / 16 / 128); ++i) {
            const uint32_t off = (uint32_t)(i * 128 + tid) * 16u;
            const float4 v = ld_shared_v4f(raw + C::kRawLat + C::kRawSc + off);
            st_shared_v4(slot + 4 * kKChunk + off, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                         __float_as_uint(v.w));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(C::B_FULL + s));
          mbar_arrive(bar(C::B_REMPTY + rs));
        }
        ms.prefetch(p, t);
      }
    }
    if (__any_sync(0xffffffffu, !(sc_max <= 146.0f) || ue_max > 134u) && lane == 0) atomicOr(p.status, STATUS_RANGE);
  } else if (ok && lane == 0 && (warp == 1 || warp == C::kPvWarp)) {
    // ---------------- UMMA issue ----------------
    // 16-bit operand type of the latent QK^T / P.V (fp16 for fp16 and FP8
    // caches) and of the RoPE QK^T (the cache's RoPE dims: bf16 unless fp16)
    constexpr bool kLatBf16 = C::kLatBf16;
    constexpr uint32_t idesc_qk = idesc_f16(128, 64, kLatBf16, false, false);
    constexpr uint32_t idesc_qr = idesc_f16(128, 64, !kFp16, false, false);
    constexpr uint32_t idesc_pv = idesc_f16(128, 256, kLatBf16, false, true);
    // descriptors: +2 in the low word advances the start address by 32 B (16
    // elements of K), +128 by 2048 B (16 tokens of the MN-major V operand)
    const uint64_t d_qr = sdesc_sw64(sb + C::OFF_QR, 16, 512);
    // S[g&1] = Q K^T over this CTA's 256 latent + 32 RoPE dims of tile g
    auto issue_qk = [&](int g) {
      const int s = g % NS;
      const uint32_t dS = tmem + kColS;
      const uint32_t slot = sb + C::OFF_RING + s * C::kSlotBytes;
      const uint64_t d_k = sdesc_sw128(slot, 16, 1024);
      const uint64_t d_kr = sdesc_sw64(slot + 4 * kKChunk, 16, 512);
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(dS, tmem + kColQ + 32u * ci + 8u * k, d_k + (uint64_t)(ci * (kKChunk >> 4) + 2 * k), idesc_qk,
                  (ci | k) ? 1u : 0u);
      }
      if constexpr (!kV41) {  // + this CTA's 32 RoPE dims
        umma_ss(dS, d_qr, d_kr, idesc_qr, 1u);
        umma_ss(dS, d_qr + 2, d_kr + 2, idesc_qr, 1u);
      }
      umma_commit(bar(C::B_SFULL));
    };
    // O[:, this CTA's 256 dims] (+)= P V of tile g; frees P and the ring slot
    auto issue_pv = [&](int g, bool first) {
      const uint64_t d_v = sdesc_sw128(sb + C::OFF_RING + (g % NS) * C::kSlotBytes, kKChunk, 1024);
      const uint32_t tp = tmem + kColP + 32u * (uint32_t)(g & 1);  // P as the A operand, from TMEM
      umma_ts(tmem, tp, d_v, idesc_pv, first ? 0u : 1u);
      umma_ts(tmem, tp + 8u, d_v + 128, idesc_pv, 1u);
      umma_ts(tmem, tp + 16u, d_v + 256, idesc_pv, 1u);
      umma_ts(tmem, tp + 24u, d_v + 384, idesc_pv, 1u);
      umma_commit(bar(C::B_PEMPTY + (g & 1)));
      umma_commit(bar(C::B_EMPTY + g % NS));
    };
    uint32_t drain_bar = bar(C::B_DRAIN);
    // Two issuing threads: warp 1 issues QK^T, warp kPvWarp issues P . V, so a
    // P . V (on the pair's critical path) never queues behind the issue of
    // a whole QK^T tile. Each waits only on its own inputs.
    PieceIter it(p, part);
    Piece pc;
    int g = 0, k = 0;
    bool failed = false;
    if (warp == 1) {
      while (!failed && it.next(pc)) {
        if (!wait(bar(C::B_QFULL), k & 1, guard)) break;
        for (int t = pc.t0; t < pc.t1; ++t, ++g) {
          if (!wait(bar(C::B_FULL + g % NS), (g / NS) & 1, guard) ||
              !wait(bar(C::B_SEMPTY), (g & 1) ^ 1, guard)) {
            failed = true;
            break;
          }
          tc_fence_after();
          *qk_started = (uint32_t)g + 1u;
          issue_qk(g);
        }
        if (failed) break;
        umma_commit(bar(C::B_QEMPTY));
        ++k;
      }
    } else {
      drain_bar = bar(C::B_DRAIN2);
      while (!failed && it.next(pc)) {
        for (int t = pc.t0; t < pc.t1; ++t, ++g) {
          // a piece's first P . V overwrites O: the previous piece's epilogue must have read it
          if (!wait(bar(C::B_PFULL + (g & 1)), (g >> 1) & 1, guard) ||
              (t == pc.t0 && k > 0 && !wait(bar(C::B_OEMPTY), (k - 1) & 1, guard))) {
            failed = true;
            break;
          }
          // The tensor pipe runs MMAs in issue order, and S of the QK^T in
          // flight is on the loop QK^T -> E reads S -> next QK^T. So P . V
          // waits for that S to complete and fills the gap while the E warps
          // read it. S(n-1) is complete once its phase is seen or once QK^T n
          // has started (it waits for S(n-1) to be read); the wait is
          // bounded, and giving up only changes the order of the MMAs. (The
          // sparse mode, bound by its gathers and dequantisation, measured
          // faster without it.)
          const uint32_t n = *qk_started;
          if (!kSparse && n > 0u) {
            const uint64_t t_0 = cycles();
            while (!mbar_test(bar(C::B_SFULL), (n - 1u) & 1u) && *qk_started == n && cycles() - t_0 < 20000u) {}
          }
          tc_fence_after();
          issue_pv(g, t == pc.t0);
        }
        ++k;
      }
    }
    // every UMMA this thread issued has completed before TMEM is released
    umma_commit(drain_bar);
    const uint64_t t_0 = cycles();
    while (!mbar_try_wait(drain_bar, 0) && cycles() - t_0 < kDrainLimitCycles) {}
  } else if (ok && warp >= 4 && warp < 8) {
    // ---------------- E warps: S -> E = exp2(x - m_own), stage, send ----------------
    const int h = 32 * (warp - 4) + lane;                 // head = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp - 4)) << 16);
    const uint32_t xr_remote = mapa(sb + C::OFF_XR, peer);
    const uint32_t xfull_remote = mapa(bar(C::B_XFULL), peer);
    const float sl2 = p.scale_log2;
    // copy this CTA's 256 latent dims of every head's query row into TMEM
    auto load_q = [&](const Piece& q_pc, int q_idx) -> bool {
      if (q_idx > 0 && !warp_ok(wait(bar(C::B_QEMPTY), (q_idx - 1) & 1, guard))) return false;
      const int b = q_pc.v % p.batch, i = q_pc.v / p.batch;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) +
                                                        ((int64_t)(b * p.s_q + i) * 128 + h) * kDQ + 256 * rank);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[64];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint4 x = __ldg(src + 16 * half + k);
          r[4 * k] = x.x; r[4 * k + 1] = x.y; r[4 * k + 2] = x.z; r[4 * k + 3] = x.w;
        }
        if constexpr (kQuant) {  // latent operands of quantised rows are fp16
          float qmax = 0.f;
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            const float x0 = __uint_as_float(r[k] << 16), x1 = __uint_as_float(r[k] & 0xFFFF0000u);
            qmax = fmaxf(qmax, fmaxf(fabsf(x0), fabsf(x1)));
            r[k] = pack_f16x2_sat(x0, x1);
          }
          // beyond fp16's largest finite value the query was saturated
          if (qmax > 65504.f) atomicOr(p.status, STATUS_RANGE);
        }
        tc_fence_after();
        tmem_st32(tl + kColQ + 64u * half, r);
        tmem_st32(tl + kColQ + 64u * half + 32u, r + 32);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_QFULL));
      return true;
    };
    PieceIter it(p, part);
    Piece pc;
    int g = 0, qi = 0;
    bool failed = false;
    while (!failed && it.next(pc)) {
      if (!load_q(pc, qi++)) break;
      MaskStream<kSparse> ms;
      ms.start(p, pc);
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        const uint64_t vm = ms.next(p, t, rank == 0 && warp == 4);
        if (!warp_ok(wait(bar(C::B_SFULL), g & 1, guard))) { failed = true; break; }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(tl + kColS, sr);
        tmem_ld32(tl + kColS + 32u, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_SEMPTY));
        // row max of the raw scores (the scale is positive, so it commutes
        // with the max); masked tokens become -inf (their rows may hold NaN)
        if (vm != ~0ull) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (!((vm >> k) & 1ull)) sr[k] = 0xFF800000u;  // -inf
        }
        const float m_own = tree_max64([&](int k) { return __uint_as_float(sr[k]); }) * sl2;
        // E = 2^(s - m_own + kEShift): fp16's normal range holds 28 binades
        // below the half's maximum and its subnormals keep an absolute
        // precision of 2^-25 below that
        const float nref = m_own == -INFINITY ? 0.f : kEShift - m_own;
        // the exponents two tokens per instruction (packed fp32 pairs)
        const uint64_t sl2_2 = f2_pack(sl2, sl2), nref2 = f2_pack(nref, nref);
        uint32_t e[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float2 x = f2_unpack(
              f2_fma(f2_pack(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])), sl2_2, nref2));
          e[u] = pack_f16x2(exp2_approx(x.x), exp2_approx(x.y));
        }
        // XS is free once this CTA's P warps have read tile g-1 from it and the
        // peer has read its copy (which frees the peer's receive buffer too)
        if (!warp_ok(wait(bar(C::B_XSFREE), (g & 1) ^ 1, guard)) ||
            !warp_ok(wait_cluster(bar(C::B_XEMPTY), (g & 1) ^ 1, guard))) {
          failed = true;
          break;
        }
        const uint32_t xs = sb + C::OFF_XS;
        const uint32_t xs_row = xs + h * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(xs_row + ((u ^ (h & 7)) << 4), e[4 * u], e[4 * u + 1], e[4 * u + 2], e[4 * u + 3]);
        reinterpret_cast<float*>(smem + C::OFF_XS + kXM)[h] = m_own;
        if (h == 0) *reinterpret_cast<uint64_t*>(smem + C::OFF_XS + kXMask) = vm;
        fence_proxy_async_smem();
        named_sync(kEBar, 128);
        if (h == 0) {
          bulk_copy_to_peer(xr_remote, xs, kXBytes, xfull_remote);
          mbar_arrive(bar(C::B_XSFULL));
        }
        ms.prefetch(p, t);
      }
    }
  } else if (ok && warp >= 8 && warp < 12) {
    // ---------------- P warps: receive, P = E_own * E_peer * 2^(m_own + m_peer - m_ref) ----------------
    const int h = 32 * (warp - 8) + lane;                 // head = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp - 8)) << 16);
    const uint32_t xr_row = sb + C::OFF_XR + h * 128;
    const uint32_t xempty_remote = mapa(bar(C::B_XEMPTY), peer);
    const float* xr_m = reinterpret_cast<const float*>(smem + C::OFF_XR + kXM);
    const int pid = threadIdx.x - 256;                    // 0..127 among P threads
    PieceIter it(p, part);
    Piece pc;
    int g = 0, pcount = 0;
    bool failed = false;
    while (!failed && it.next(pc)) {
      const int b = pc.v % p.batch, i = pc.v / p.batch;
      float m = -INFINITY, l = 0.f;
      for (int t = pc.t0; t < pc.t1; ++t, ++g) {
        // (1) this CTA's own E and m of tile g, staged by the E warps (always
        // before the peer's copy of the same tile lands, so read first)
        uint32_t ep[32], eo[32];
        if (!warp_ok(wait(bar(C::B_XSFULL), g & 1, guard))) { failed = true; break; }
        const uint32_t xs_row = sb + C::OFF_XS + h * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 o = ld_shared_v4f(xs_row + ((u ^ (h & 7)) << 4));
          eo[4 * u] = __float_as_uint(o.x); eo[4 * u + 1] = __float_as_uint(o.y);
          eo[4 * u + 2] = __float_as_uint(o.z); eo[4 * u + 3] = __float_as_uint(o.w);
        }
        const float m_own = reinterpret_cast<const float*>(smem + C::OFF_XS + kXM)[h];
        const uint64_t vm = *reinterpret_cast<const volatile uint64_t*>(smem + C::OFF_XS + kXMask);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_XSFREE));
        // (2) the peer's E and m of tile g
        if (pid == 0) mbar_arrive_expect_tx(bar(C::B_XFULL), kXBytes);
        if (!warp_ok(wait_cluster(bar(C::B_XFULL), g & 1, guard))) { failed = true; break; }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 o = ld_shared_v4f(xr_row + ((u ^ (h & 7)) << 4));
          ep[4 * u] = __float_as_uint(o.x); ep[4 * u + 1] = __float_as_uint(o.y);
          ep[4 * u + 2] = __float_as_uint(o.z); ep[4 * u + 3] = __float_as_uint(o.w);
        }
        const float m_peer = xr_m[h];
        {
          // Hand the receive buffer back to the peer. The arrive is relaxed,
          // so it must not be performed before this warp's loads from the
          // buffer have returned: its address depends on every loaded value
          // (through a mask that is zero at run time, the rank being 0 or 1).
          uint32_t dep = __float_as_uint(m_peer);
#pragma unroll
          for (int u = 0; u < 8; ++u) dep |= ep[4 * u];
          dep = __reduce_or_sync(0xffffffffu, dep) & (rank >> 1);
          if (lane == 0) mbar_arrive_remote_relaxed(xempty_remote + dep);
        }
        // (3) P = 2^(s - m_use) against the running reference max m_use,
        // moved lazily (P <= 256). mt = m_own + m_peer bounds the tile's row
        // max from above, far above it when the halves peak on different
        // tokens. S = sum of the products certifies the row (kCertify).
        const float mt = m_own + m_peer;
        // the products E_own E_peer of a token pair, up to 2^(2 kEShift), in
        // one mixed-precision fma each (exact, and the same in both CTAs)
        auto prod = [&](int u) { return mul_f16x2_to_f32(eo[u], ep[u]); };
        float m_use, alpha, rs0;
        bool resc, cert;
        if constexpr (C::kLatBf16) {
          // bf16 P keeps fp32's exponent range: the reference may sit far
          // above the tile's row max, so take mt and go in one pass
          const RowRef r(m, mt);
          m_use = r.m_use;
          alpha = r.alpha;
          resc = r.resc;
          const float cf = r.live ? exp2_approx((mt - m_use) - 2.f * kEShift) : 0.f;
          // P and the row sum two tokens per instruction (packed fp32 pairs;
          // four partial sums keep the dependency chains short)
          const uint64_t cf2 = f2_pack(cf, cf);
          uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float2 e = prod(u);
            const uint64_t p2 = f2_mul(f2_pack(e.x, e.y), cf2);
            rs2[u & 3] = f2_add(rs2[u & 3], p2);
            const float2 pp = f2_unpack(p2);
            ep[u] = pack_bf16x2(pp.x, pp.y);
          }
          const float2 r01 = f2_unpack(f2_add(f2_add(rs2[0], rs2[1]), f2_add(rs2[2], rs2[3])));
          rs0 = r01.x + r01.y;
          // (cf = 0: no valid token, or a tile more than 2^126 below the row)
          cert = !(cf > 0.f) || rs0 >= kCertify * cf;
        } else {
          // fp16 P ends at 2^-24: the reference comes from S, which puts the
          // tile's row max within 6 binades: mt - 2 kEShift + log2 S - 6 <= Mt
          uint64_t a2[32];
          uint64_t sv2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float2 e = prod(u);
            a2[u] = f2_pack(e.x, e.y);
            sv2[u & 3] = f2_add(sv2[u & 3], a2[u]);
          }
          const float2 s01 = f2_unpack(f2_add(f2_add(sv2[0], sv2[1]), f2_add(sv2[2], sv2[3])));
          const float S = s01.x + s01.y;
          const RowRef r(m, (mt == -INFINITY || !(S > 0.f)) ? -INFINITY : mt + (log2_approx(S) - 2.f * kEShift));
          m_use = r.m_use;
          alpha = r.alpha;
          resc = r.resc;
          const float cf = r.live ? exp2_approx((mt - m_use) - 2.f * kEShift) : 0.f;
          const uint64_t cf2 = f2_pack(cf, cf);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float2 pp = f2_unpack(f2_mul(a2[u], cf2));
            ep[u] = pack_f16x2(pp.x, pp.y);
          }
          rs0 = S * cf;
          cert = !r.live || S >= kCertify;
        }
        {
          // The halves disagree by more than about 22 binades on a row
          // (rare): the row's result from here on is not certified. For
          // 16-bit caches the row is flagged, and the combine kernel
          // recomputes it exactly from q and the cache rows; quantised rows
          // report it. (Kept out of this kernel: its slow path would cost the common
          // one registers and code.)
          const uint32_t unc = __ballot_sync(0xffffffffu, !cert);
          if (unc != 0u && rank == 0 && lane == 0) {
            if constexpr (kQuant) atomicOr(p.status, STATUS_RANGE);
            else atomicOr(p.exact_flags + (int64_t)pc.v * 4 + (warp - 8), unc);
          }
        }
        l = l * alpha + rs0;
        m = m_use;
        // a rescale of O needs every earlier P . V done; they complete in issue
        // order, so waiting for tile g-1 is enough
        if (__any_sync(0xffffffffu, resc) && t != pc.t0) {
          if (!warp_ok(wait(bar(C::B_PEMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1, guard))) { failed = true; break; }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t r[32];
            tmem_ld32(tl + 32u * cc, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
            tmem_st32(tl + 32u * cc, r);
          }
          tmem_wait_st();
        }
        if (!kQuant && vm != ~0ull) {
          // zero the V rows of masked tokens: 0 * (whatever is there) must not
          // turn into NaN inside P . V (the dequant warps do this for quantised rows)
          const uint32_t slot = sb + C::OFF_RING + (g % NS) * C::kSlotBytes;
          for (int e2 = pid; e2 < 64 * 32; e2 += 128) {
            const int row = e2 >> 5, u = e2 & 31;
            if (!((vm >> row) & 1ull))
              st_shared_v4(slot + (u >> 3) * kKChunk + row * 128 + (u & 7) * 16, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // P of tile g into TMEM buffer g&1 (the A operand of P . V), once P . V
        // of tile g-2 is done with that buffer
        if (!warp_ok(wait(bar(C::B_PEMPTY + (g & 1)), ((g >> 1) & 1) ^ 1, guard))) { failed = true; break; }
        tc_fence_after();
        tmem_st32(tl + kColP + 32u * (uint32_t)(g & 1), ep);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PFULL + (g & 1)));
      }
      if (failed) break;
      // ---- epilogue of the piece: O / l -> out (single piece) or partial ----
      // (P . V of the piece's last tile completes after every earlier one)
      if (!warp_ok(wait(bar(C::B_PEMPTY + ((g - 1) & 1)), ((g - 1) >> 1) & 1, guard))) { failed = true; break; }
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      const int64_t row = (int64_t)(b * p.s_q + i) * 128 + h;
      // each thread writes 32 consecutive values of its own row per chunk;
      // 32-byte stores make every request of a warp a whole sector, and the
      // TMEM load of chunk cc+1 is in flight while chunk cc is stored
      const uint64_t inv2 = f2_pack(inv_l, inv_l);
      auto store_chunk = [&](int cc, uint32_t* r) {
        if (pc.fin) {
          OutT* dst = reinterpret_cast<OutT*>(p.out) + row * kDV + 256 * rank + 32 * cc;
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 ac = f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])), inv2));
            w[k] = kFp16 ? pack_f16x2(ac.x, ac.y) : pack_bf16x2(ac.x, ac.y);
          }
          if (p.out_v8) {
            st_global_v8(dst, w);
            st_global_v8(dst + 16, w + 8);
          } else {
#pragma unroll
            for (int k = 0; k < 16; k += 4)
              *reinterpret_cast<uint4*>(dst + 2 * k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
          }
        } else {
          const int d0 = 256 * (int)rank + 32 * cc;
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 ac = f2_unpack(f2_mul(f2_pack(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), inv2));
            r[k] = __float_as_uint(ac.x);
            r[k + 1] = __float_as_uint(ac.y);
          }
#pragma unroll
          for (int k = 0; k < 32; k += 8) st_global_v8(p.o_part + opart_index(pc.split, 128, h, d0 + k), r + k);
        }
      };
      uint32_t ra[32], rb[32];
      tmem_ld32(tl, ra);
      tmem_wait_ld();
      pin_regs32(ra);
#pragma unroll 1
      for (int cc = 0; cc < 8; cc += 2) {
        tmem_ld32(tl + 32u * (cc + 1), rb);
        store_chunk(cc, ra);
        tmem_wait_ld();
        pin_regs32(rb);
        if (cc + 2 < 8) tmem_ld32(tl + 32u * (cc + 2), ra);
        store_chunk(cc + 1, rb);
        tmem_wait_ld();
        pin_regs32(ra);
      }
      if (rank == 0) {
        if (pc.fin) p.lse[row] = lse;
        else p.lse_part[(int64_t)pc.split * 128 + h] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
      ++pcount;
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
