// params.h -- kernel parameter blocks and the metadata layout shared by the
// host entry points and the kernels.
#pragma once
#include <cstdint>

namespace mla {

constexpr int kTile = 64;         // tokens per KV tile (= page_block)
constexpr int kDK = 576;          // latent 512 + RoPE 64
constexpr int kDV = 512;
constexpr int kRowBytesFp8 = 656;
constexpr int kDV41 = 512;        // V4.1 rows: 512 values (latent and RoPE together)
constexpr int kRowBytesFp8_528 = 528;
constexpr int kRowBytesFp4_288 = 288;
// schedule cost of starting a request, in tiles: a piece switch of the
// 128-head kernel (a 256 KB epilogue, the next query, refilling the pair's
// pipeline) costs more than one of the 16-head kernel
constexpr int kPieceOverhead = 5;
constexpr int kPieceOverheadFewHeads = 2;

// ---- metadata (int32 words) ----
// header
enum : int {
  H_MAGIC = 0, H_BATCH, H_SQ, H_HQ, H_TOPK, H_KVFMT, H_CAUSAL, H_PAGE, H_PARTS, H_HASH,
  H_NPIECES, H_VREQ, H_WORDS = 16
};
constexpr int32_t kMetaMagic = 0x31414C4D;  // "MLA1"
// one record per SM part: first piece (v, tile), end (v, tile exclusive),
// split ordinal of the first piece
enum : int { P_BV = 0, P_BT, P_EV, P_ET, P_SPLIT, P_WORDS = 8 };

__host__ __device__ inline int meta_words(int vreq, int parts) {
  (void)vreq;
  return H_WORDS + parts * P_WORDS;
}

// hash of the per-request lengths (or topk) baked into the metadata so the
// decode kernel can tell that it is being reused for a different problem
__host__ __device__ inline uint32_t hash_step(uint32_t h, uint32_t x) {
  h ^= x + 0x9E3779B9u + (h << 6) + (h >> 2);
  return h;
}

// ---- workspace ----
// [0, 256): status word; then o_part fp32 [max_splits][64][h_q][8] (opart_index); then
// lse_part fp32 [max_splits, h_q]; then the exact-recompute flags uint32
// [vreq][4]: one bit per head (h_q <= 128), set by the decode kernel for a row
// it could not certify and cleared by the combine kernel once it has
// recomputed that row exactly (zero between calls)
constexpr size_t kWsHeader = 256;
// o_part element (split, head h, dim d): [split][64 units of 8 dims][h_q][8],
// so that a warp of consecutive heads stores one unit as one contiguous run
// (1 KB for 32 heads) and the combine reads 16 heads' unit as 512 B
__host__ __device__ inline int64_t opart_index(int64_t split, int h_q, int h, int d) {
  return ((split * 64 + (d >> 3)) * h_q + h) * 8 + (d & 7);
}
__host__ __device__ inline int64_t max_splits(int vreq, int parts) { return (int64_t)vreq + parts; }
__host__ __device__ inline size_t ws_flags_offset(int vreq, int parts, int h_q) {
  const int64_t S = max_splits(vreq, parts);
  return kWsHeader + (size_t)S * h_q * 512 * sizeof(float) + (size_t)S * h_q * sizeof(float);
}
__host__ __device__ inline size_t ws_bytes(int vreq, int parts, int h_q) {
  return ws_flags_offset(vreq, parts, h_q) + (size_t)vreq * 4 * sizeof(uint32_t);
}

struct MetaParams {
  const int32_t* seqlens;   // [batch] or null (sparse)
  int batch, s_q, h_q, topk, kv_format, causal, page_block, parts;
  int32_t* meta;
  int32_t* split_off;       // [vreq + 1]
};

struct DecodeParams {
  const void* q;               // [batch, s_q, h_q, 576] (512 for the V4.1 rows)
  const int32_t* block_table;  // [batch, max_blocks] (dense)
  const int32_t* seqlens;      // [batch]
  const int32_t* indices;      // [batch, s_q, topk] (sparse) or null
  const uint8_t* kv;           // the cache rows as bytes (1152-B 16-bit, or 656-, 528- or 288-B quantised rows)
  const int32_t* meta;
  const int32_t* split_off;
  void* out;                   // [batch, s_q, h_q, 512], q dtype
  float* lse;                  // [batch, s_q, h_q]
  float* o_part;               // [max_splits][64 units][h_q][8] (opart_index)
  float* lse_part;             // [max_splits, h_q]
  uint32_t* status;
  uint32_t* exact_flags;       // [vreq][4] head bits of rows to recompute exactly
  int64_t num_blocks;
  int64_t num_rows;            // num_blocks * page_block
  int max_blocks;
  int batch, s_q, h_q, topk, causal, kv_format, parts;
  int out_v8;                  // out is 32-B aligned: 32-byte stores in the epilogue
  float scale_log2;            // softmax_scale * log2(e)
  // test hook, 0 in normal use: before any copy is issued, thread 0 of each CTA
  // waits this many cycles on a barrier that nothing arrives at, so the wait
  // gives up, reports STATUS_TIMEOUT and the CTA skips all work
  uint32_t stall_cycles;
};

struct CombineParams {
  const int32_t* split_off;
  const float* o_part;
  const float* lse_part;
  void* out;
  float* lse;
  int batch, s_q, h_q;
  int fp16;
  // exact recompute of the rows the decode kernel flagged (dense 16-bit
  // caches; null otherwise): q, the cache rows (1152 B each), block table and
  // lengths of the call
  uint32_t* exact_flags;
  const void* q;
  const uint8_t* kv;
  const int32_t* block_table;
  const int32_t* seqlens;
  int64_t num_blocks;
  int max_blocks, causal;
  float scale_log2;
};

}  // namespace mla
