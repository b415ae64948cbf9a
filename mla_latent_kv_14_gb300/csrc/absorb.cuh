// absorb.cuh -- the two per-head GEMMs around the decode kernel, sm_103a.
//
// Weight absorption ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §六 '吸收'):
// the key up-projection W^UK_i (d_h x d_c) folds into the query side,
//     q~_{t,i} = W^UK_i^T q^C_{t,i}          (d_c = 512 wide),
// so every head scores the shared latent row; and the value up-projection
// W^UV_i (d_h x d_c) is applied once to the attention-weighted latent,
//     o_{t,i}  = W^UV_i  o~_{t,i}             (d_h = 128 wide).
// Both are, per head, a GEMM over the T query tokens:
//     absorb:     Q~_i [T x 512] = Q^C_i [T x 128] . W^UK_i [128 x 512]
//     up-project: O_i  [T x 128] = O~_i  [T x 512] . W^UV_i^T [512 x 128]
//
// One CTA per (head, 128-token tile), 128 threads. Thread 0 loads both
// operands with one TMA box each (4-D tensor maps that pick the head and lay
// the tile out chunk-major, 128-byte swizzled) and issues single-CTA UMMAs
// (M = 128 tokens) into TMEM; the four warps then read their 32 token rows
// back and store them as 16-bit values. Tokens past T are zero-filled by the
// copy and not stored. Every wait is bounded; a wait that gives up sets the
// status word (if one is given) and nothing is stored. A copy whose wait gave
// up is waited for once more before the CTA exits. `stall` (a test hook, 0 in
// normal use) makes thread 0 first wait that many cycles on a barrier nothing
// arrives at, so the wait gives up before any copy is issued.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mla {
namespace absorb {

constexpr int kThreads = 128;
constexpr int kTokTile = 128;
constexpr int kChunk = 128 * 128;  // one 64-wide chunk of 128 rows, 16-bit: 16 KB
constexpr uint64_t kLimit = 2000000000ull;

// 32 fp32 of one row -> 16-bit values at dst (16-B aligned)
template <bool kFp16>
__device__ __forceinline__ void store_row32(void* dst, const uint32_t* r) {
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float a = __uint_as_float(r[2 * k]), c = __uint_as_float(r[2 * k + 1]);
    w[k] = kFp16 ? pack_f16x2(a, c) : pack_bf16x2(a, c);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) d[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit = kLimit) {
  const uint64_t t0 = cycles();
  while (!mbar_try_wait(bar, parity))
    if (cycles() - t0 > limit) return false;
  return true;
}

// Q~ [T, h, 576] dims [0, 512) = per head Q^C [T, h, 128] . W^UK [h, 128, 512].
// tm_a: dims {64, T, 2, h} of q_nope; tm_b: dims {64, 128, 8, h} of w_uk.
constexpr uint32_t kAbsorbSmem = 2 * kChunk + 8 * kChunk + 64 + 1024;

template <bool kFp16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_absorb_q_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        void* q_out, int T, int h, uint32_t* status, uint32_t stall) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t a_s = sb, b_s = sb + 2 * kChunk;
  const uint32_t bar_full = sb + 10 * kChunk, bar_done = bar_full + 8, bar_stall = bar_full + 32;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + 10 * kChunk + 16);
  const int head = blockIdx.x, t0 = blockIdx.y * kTokTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_done, 1);
    mbar_init(bar_stall, 1);
    misc[1] = 1u;  // ok
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(misc)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (threadIdx.x == 0 && stall && !wait_bounded(bar_stall, 0, stall)) {
    misc[1] = 0u;  // test hook: nothing is issued
    if (status) atomicOr(status, STATUS_TIMEOUT);
    umma_commit(bar_done);
  } else if (threadIdx.x == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    mbar_arrive_expect_tx(bar_full, 10 * kChunk);
    tma_load_4d(a_s, &tm_a, bar_full, 0, t0, 0, head);
    tma_load_4d(b_s, &tm_b, bar_full, 0, 0, 0, head);
    if (!wait_bounded(bar_full, 0)) {
      misc[1] = 0u;
      if (status) atomicOr(status, STATUS_TIMEOUT);
      (void)wait_bounded(bar_full, 0);  // do not exit with the copy in flight
    } else {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_f16(128, 256, !kFp16, false, true);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        // A: K-major, chunk kk/4, 16 elements (32 B) per step inside it
        const uint64_t da = sdesc_sw128(a_s + (kk >> 2) * kChunk, 16, 1024) + 2 * (kk & 3);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          // B: N-major, 64-wide chunks kChunk apart, 16 rows of K (2 KB) per step
          const uint64_t db = sdesc_sw128(b_s + 4 * j * kChunk, kChunk, 1024) + 128 * kk;
          umma_ss(tmem + 256u * j, da, db, idesc, kk > 0 ? 1u : 0u);
        }
      }
    }
    umma_commit(bar_done);  // also arrives when no MMA was issued
  }
  __syncwarp();
  const bool done = __all_sync(0xffffffffu, wait_bounded(bar_done, 0));
  tc_fence_after();
  // tcgen05.ld is warp-collective: the whole warp loads, each lane stores
  // only its own token
  const int t = t0 + 32 * warp + lane;
  if (done && misc[1] && t0 + 32 * warp < T) {
    uint8_t* row = reinterpret_cast<uint8_t*>(q_out) + ((int64_t)t * h + head) * 576 * 2;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int cc = 0; cc < 16; ++cc) {
      uint32_t r[32];
      tmem_ld32(tl + 32u * cc, r);
      tmem_wait_ld();
      if (t < T) store_row32<kFp16>(row + 64 * cc, r);
    }
  } else if (!done && threadIdx.x == 0 && status) {
    atomicOr(status, STATUS_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// O [T, h, 128] = per head O~ [T, h, 512] . W^UV [h, 128, 512]^T, the 512-wide
// contraction in two halves through one 128 KB buffer.
// tm_a: dims {64, T, 8, h} of o_lat; tm_b: dims {64, 128, 8, h} of w_uv.
constexpr uint32_t kUpSmem = 8 * kChunk + 64 + 1024;  // + barriers and the TMEM slot

template <bool kFp16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_up_project_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                          void* o_out, int T, int h, uint32_t* status, uint32_t stall) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t a_s = sb, b_s = sb + 4 * kChunk;
  // bar_done + 8*half: the MMAs of that half of the contraction are done
  const uint32_t bar_full = sb + 8 * kChunk, bar_done = bar_full + 8, bar_stall = bar_full + 40;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + 8 * kChunk + 24);
  const int head = blockIdx.x, t0 = blockIdx.y * kTokTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_done, 1);
    mbar_init(bar_done + 8, 1);
    mbar_init(bar_stall, 1);
    misc[1] = 1u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(misc)), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    constexpr uint32_t idesc = idesc_f16(128, 128, !kFp16, false, false);
    // test hook: a wait that gives up before anything is issued
    bool ok = !(stall && !wait_bounded(bar_stall, 0, stall));
    for (int half = 0; half < 2 && ok; ++half) {
      // the buffer is free once the first half's MMAs are done
      if (half == 1 && !wait_bounded(bar_done, 0)) { ok = false; break; }
      mbar_arrive_expect_tx(bar_full, 8 * kChunk);
      tma_load_4d(a_s, &tm_a, bar_full, 0, t0, 4 * half, head);
      tma_load_4d(b_s, &tm_b, bar_full, 0, 0, 4 * half, head);
      if (!wait_bounded(bar_full, half)) {
        ok = false;
        (void)wait_bounded(bar_full, half);  // do not exit with the copy in flight
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        // both operands K-major: chunk kk/4, 32 B per step inside it
        const uint64_t da = sdesc_sw128(a_s + (kk >> 2) * kChunk, 16, 1024) + 2 * (kk & 3);
        const uint64_t db = sdesc_sw128(b_s + (kk >> 2) * kChunk, 16, 1024) + 2 * (kk & 3);
        umma_ss(tmem, da, db, idesc, (half | kk) ? 1u : 0u);
      }
      umma_commit(bar_done + 8u * half);
    }
    if (!ok) {
      misc[1] = 0u;
      if (status) atomicOr(status, STATUS_TIMEOUT);
      umma_commit(bar_done + 8);  // lets the epilogue's wait end once earlier MMAs are done
    }
  }
  __syncwarp();
  const bool done = __all_sync(0xffffffffu, wait_bounded(bar_done + 8, 0));
  tc_fence_after();
  const int t = t0 + 32 * warp + lane;
  if (done && misc[1] && t0 + 32 * warp < T) {   // warp-uniform: tcgen05.ld is warp-collective
    uint8_t* row = reinterpret_cast<uint8_t*>(o_out) + ((int64_t)t * h + head) * 128 * 2;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t r[32];
      tmem_ld32(tl + 32u * cc, r);
      tmem_wait_ld();
      if (t < T) store_row32<kFp16>(row + 64 * cc, r);
    }
  } else if (!done && threadIdx.x == 0 && status) {
    atomicOr(status, STATUS_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace absorb
}  // namespace mla
