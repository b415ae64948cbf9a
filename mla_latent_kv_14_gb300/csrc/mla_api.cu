// mla_api.cu -- the C ABI declared in include/mla.h: argument checks, tensor
// maps, launches. Every argument check happens before anything is enqueued.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/mla.h"
#include "absorb.cuh"
#include "decode_dense.cuh"
#include "decode_fewheads.cuh"
#include "params.h"
#include "quant.cuh"
#include "sched.cuh"

using namespace mla;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kFewHeads = few::kNH;  // query heads of the transposed few-heads kernel

mla_status cuda_fail(cudaError_t e) {
  (void)cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

#define MLA_CUDA(x)                              \
  do {                                           \
    cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    (void)cudaGetLastError();
  });
  return fn;
}

// 2-D row-major tensor [rows, cols] of `elem` bytes, box [box_rows, box_cols]
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, uint64_t rows, uint64_t cols,
              uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  (void)elem;
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows, 576] 16-bit tensor seen as [rows][9 chunks of 64 dims]: dims {64,
// rows, 9} with chunk stride 128 B; one box = box_rows rows x box_chunks chunks,
// laid out in shared memory chunk-major (128-B swizzled 64-dim rows).
bool make_map_chunks(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t rows, uint32_t box_rows,
                     uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, 9};
  cuuint64_t strides[2] = {kDK * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D 16-bit tensor map with 128-byte swizzle (the inner box is 64
// elements = 128 B); strides in bytes for dims 1..3.
bool make_map_4d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, const cuuint64_t (&dims)[4],
                 const cuuint64_t (&strides)[3], const cuuint32_t (&box)[4]) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// test hook (mla_set_test_stall): cycles the next launches wait on a barrier
// nothing arrives at before giving up; 0 in normal use
std::atomic<uint32_t> g_test_stall{0};

// per-device number of co-resident 2-CTA clusters of the 128-head decode
// kernel, and of co-resident CTAs of the few-heads kernel
std::atomic<int> g_parts[kMaxDevices];
std::atomic<int> g_parts_few[kMaxDevices];
std::once_flag g_attr_once[kMaxDevices];

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int kMode>
cudaError_t set_mode_smem() {
  return set_smem(dense::mla_decode_kernel<kMode>, dense::Cfg<kMode>::kSmemBytes);
}

cudaError_t prepare_device(int dev) {
  cudaError_t err = cudaSuccess;
  std::call_once(g_attr_once[dev], [&] {
    err = set_mode_smem<dense::MODE_BF16>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_FP16>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_FP8>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_FP8_SPARSE>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_V41_FP8>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_V41_FP8_SPARSE>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_V41_FP4>();
    if (err == cudaSuccess) err = set_mode_smem<dense::MODE_V41_FP4_SPARSE>();
    if (err == cudaSuccess) err = set_smem(few::mla_decode_fewheads_kernel<false>, few::kSmemBytes);
    if (err == cudaSuccess) err = set_smem(few::mla_decode_fewheads_kernel<true>, few::kSmemBytes);
    if (err == cudaSuccess) {
      int per_sm = 0, sms = 0;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, few::mla_decode_fewheads_kernel<false>,
                                                          few::kThreads, few::kSmemBytes);
      if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (err == cudaSuccess) g_parts_few[dev].store(per_sm * sms > 0 ? per_sm * sms : 1);
    }
    if (err == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(dense::kThreads, 1, 1);
      cfg.dynamicSmemBytes = dense::Cfg<dense::MODE_BF16>::kSmemBytes;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      err = cudaOccupancyMaxActiveClusters(&n, dense::mla_decode_kernel<dense::MODE_BF16>, &cfg);
      if (err == cudaSuccess) g_parts[dev].store(n > 0 ? n : 1);
    }
  });
  if (err == cudaSuccess && (g_parts[dev].load() <= 0 || g_parts_few[dev].load() <= 0))
    err = cudaErrorInitializationError;
  return err;
}

}  // namespace

extern "C" {

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported";
    case MLA_ERR_STALE_METADATA: return "metadata does not match this call (recompute it)";
    case MLA_ERR_INDEX: return "out-of-range page or index skipped";
    case MLA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_RANGE: return "a value or score beyond the range a quantised cache path certifies";
    default: return "unknown status";
  }
}

int mla_num_sm_parts(int device) {
  if (device < 0 || device >= kMaxDevices) return -1;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) { (void)cudaGetLastError(); return -1; }
  if (cur != device && cudaSetDevice(device) != cudaSuccess) { (void)cudaGetLastError(); return -1; }
  cudaError_t e = prepare_device(device);
  if (cur != device) cudaSetDevice(cur);
  if (e != cudaSuccess) { (void)cudaGetLastError(); return -1; }
  return g_parts[device].load();
}

int mla_num_sm_parts_for(int device, int h_q) {
  const int n = mla_num_sm_parts(device);
  if (n <= 0) return n;
  if (h_q == kFewHeads) return g_parts_few[device].load();
  return h_q == 128 ? n : -1;
}

size_t mla_metadata_size(int batch, int s_q, int parts) {
  if (batch <= 0 || s_q <= 0 || parts <= 0) return 0;
  return (size_t)meta_words(batch * s_q, parts) * sizeof(int32_t);
}

size_t mla_workspace_size(int batch, int s_q, int h_q, int parts) {
  if (batch <= 0 || s_q <= 0 || h_q <= 0 || parts <= 0) return 0;
  return ws_bytes(batch * s_q, parts, h_q);
}

mla_status mla_get_metadata(const int32_t* cache_seqlens, int batch, int s_q, int h_q, int h_kv, int topk,
                            int kv_format, int causal, int page_block, int parts, void* metadata, int32_t* num_splits,
                            void* stream) {
  if (batch <= 0 || s_q <= 0 || parts <= 0 || topk < 0) return MLA_ERR_INVALID_ARG;
  if (kv_format < MLA_KV_16BIT || kv_format > MLA_KV_FP4_288) return MLA_ERR_INVALID_ARG;
  if (h_kv != 1 || page_block != kTile) return MLA_ERR_INVALID_ARG;
  if (h_q != 128 && h_q != kFewHeads) return MLA_ERR_UNSUPPORTED;
  if (h_q == kFewHeads && (topk > 0 || kv_format)) return MLA_ERR_UNSUPPORTED;  // few heads: dense 16-bit caches
  if (!metadata || !num_splits) return MLA_ERR_INVALID_ARG;
  if (topk == 0 && !cache_seqlens) return MLA_ERR_INVALID_ARG;
  if (topk > 0 && causal) return MLA_ERR_INVALID_ARG;
  if ((int64_t)batch * s_q > kMaxVreq) return MLA_ERR_UNSUPPORTED;
  MetaParams mp{topk > 0 ? nullptr : cache_seqlens, batch, s_q, h_q, topk, kv_format, causal ? 1 : 0,
                page_block, parts, static_cast<int32_t*>(metadata), num_splits};
  const size_t smem = metadata_smem_bytes(batch * s_q);
  if (smem > 48 * 1024) {
    MLA_CUDA(cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  }
  // one block; small problems use fewer threads (cheaper block-wide scans)
  const int need = (batch * s_q > parts ? batch * s_q : parts);
  int threads = (need + 31) / 32 * 32;
  threads = threads < 128 ? 128 : (threads > kMetaThreads ? kMetaThreads : threads);
  // launched as a programmatic dependent of whatever precedes it on the stream
  // (e.g. the previous call's combine); the kernel waits for it before any
  // global access, so only the launch latency is overlapped
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3(1, 1, 1);
  mc.blockDim = dim3((unsigned)threads, 1, 1);
  mc.dynamicSmemBytes = smem;
  mc.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute mat[1];
  mat[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  mat[0].val.programmaticStreamSerializationAllowed = 1;
  mc.attrs = mat;
  mc.numAttrs = 1;
  MLA_CUDA(cudaLaunchKernelEx(&mc, mla_metadata_kernel, mp));
  return MLA_OK;
}

}  // extern "C"

namespace {
enum : int { STAGE_SPLIT = 1, STAGE_COMBINE = 2 };

template <int kMode>
cudaError_t launch_mode(cudaLaunchConfig_t cfg, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const CUtensorMap& d, const DecodeParams& p) {
  cfg.blockDim = dim3(dense::Cfg<kMode>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dense::Cfg<kMode>::kSmemBytes;
  return cudaLaunchKernelEx(&cfg, dense::mla_decode_kernel<kMode>, a, b, c, d, p);
}

// the 128-head decode kernel of one cache format / addressing mode
cudaError_t launch_decode_mode(int mode, const cudaLaunchConfig_t& cfg, const CUtensorMap& a, const CUtensorMap& b,
                               const CUtensorMap& c, const CUtensorMap& d, const DecodeParams& p) {
  switch (mode) {
    case dense::MODE_BF16: return launch_mode<dense::MODE_BF16>(cfg, a, b, c, d, p);
    case dense::MODE_FP16: return launch_mode<dense::MODE_FP16>(cfg, a, b, c, d, p);
    case dense::MODE_FP8: return launch_mode<dense::MODE_FP8>(cfg, a, b, c, d, p);
    case dense::MODE_FP8_SPARSE: return launch_mode<dense::MODE_FP8_SPARSE>(cfg, a, b, c, d, p);
    case dense::MODE_V41_FP8: return launch_mode<dense::MODE_V41_FP8>(cfg, a, b, c, d, p);
    case dense::MODE_V41_FP8_SPARSE: return launch_mode<dense::MODE_V41_FP8_SPARSE>(cfg, a, b, c, d, p);
    case dense::MODE_V41_FP4: return launch_mode<dense::MODE_V41_FP4>(cfg, a, b, c, d, p);
    default: return launch_mode<dense::MODE_V41_FP4_SPARSE>(cfg, a, b, c, d, p);
  }
}

// Host-side argument checks of a decode call; nothing is enqueued. The
// workspace is checked only when the caller supplies one (check_ws).
mla_status validate_decode(const void* q, int q_dtype, const void* kvcache, int64_t num_blocks, int page_block,
                           const int32_t* block_table, int max_blocks, const int32_t* cache_seqlens, int batch,
                           int s_q, int h_q, int head_dim_v, const void* metadata, const int32_t* num_splits,
                           int parts, float softmax_scale, int causal, int kv_format, const int32_t* indices, int topk,
                           void* out, float* lse, bool check_ws, void* workspace, size_t workspace_bytes) {
  if (!q || !kvcache || !out || !lse || (check_ws && !workspace) || !metadata || !num_splits)
    return MLA_ERR_INVALID_ARG;
  if (q_dtype != MLA_DTYPE_BF16 && q_dtype != MLA_DTYPE_FP16) return MLA_ERR_INVALID_ARG;
  if (kv_format < MLA_KV_16BIT || kv_format > MLA_KV_FP4_288) return MLA_ERR_INVALID_ARG;
  if (head_dim_v != kDV || page_block != kTile) return MLA_ERR_INVALID_ARG;
  if (batch <= 0 || s_q <= 0 || parts <= 0 || num_blocks <= 0 || topk < 0) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (indices && causal) return MLA_ERR_INVALID_ARG;        // the index list already fixes the key set
  if ((indices != nullptr) != (topk > 0)) return MLA_ERR_INVALID_ARG;
  if (!indices && (!block_table || max_blocks <= 0 || !cache_seqlens)) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kvcache, 16) || !aligned(out, 16) || (check_ws && !aligned(workspace, 256)) ||
      !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (check_ws && workspace_bytes < mla_workspace_size(batch, s_q, h_q, parts)) return MLA_ERR_INVALID_ARG;
  if (num_blocks * (int64_t)page_block >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
  if (h_q != 128 && h_q != kFewHeads) return MLA_ERR_UNSUPPORTED;
  if (h_q == kFewHeads && (indices || kv_format)) return MLA_ERR_UNSUPPORTED;  // few heads: dense 16-bit caches
  if (indices && !kv_format) return MLA_ERR_UNSUPPORTED;                 // token-sparse decode reads quantised rows
  if (kv_format && q_dtype != MLA_DTYPE_BF16) return MLA_ERR_UNSUPPORTED; // quantised rows pair with bf16 queries
  const int64_t qrows = (int64_t)batch * s_q * h_q;
  if (qrows >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

mla_status decode_impl(int stages, const void* q, int q_dtype, const void* kvcache, int64_t num_blocks,
                       int page_block, const int32_t* block_table, int max_blocks, const int32_t* cache_seqlens,
                       int batch, int s_q, int h_q, int head_dim_v, const void* metadata, const int32_t* num_splits,
                       int parts, float softmax_scale, int causal, int kv_format, const int32_t* indices, int topk,
                       void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  // ---- host-side argument checks (nothing is enqueued on failure) ----
  const mla_status v = validate_decode(q, q_dtype, kvcache, num_blocks, page_block, block_table, max_blocks,
                                       cache_seqlens, batch, s_q, h_q, head_dim_v, metadata, num_splits, parts,
                                       softmax_scale, causal, kv_format, indices, topk, out, lse, true, workspace,
                                       workspace_bytes);
  if (v != MLA_OK) return v;
  const int64_t qrows = (int64_t)batch * s_q * h_q;

  int dev = 0;
  MLA_CUDA(cudaGetDevice(&dev));
  if (dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  MLA_CUDA(prepare_device(dev));

  const bool fp16 = q_dtype == MLA_DTYPE_FP16;
  const bool sparse = indices != nullptr;
  const bool v41 = kv_format == MLA_KV_FP8_528 || kv_format == MLA_KV_FP4_288;
  int mode = fp16 ? dense::MODE_FP16 : dense::MODE_BF16;
  if (kv_format == MLA_KV_FP8_656) mode = sparse ? dense::MODE_FP8_SPARSE : dense::MODE_FP8;
  if (kv_format == MLA_KV_FP8_528) mode = sparse ? dense::MODE_V41_FP8_SPARSE : dense::MODE_V41_FP8;
  if (kv_format == MLA_KV_FP4_288) mode = sparse ? dense::MODE_V41_FP4_SPARSE : dense::MODE_V41_FP4;
  const CUtensorMapDataType dt = fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t kvrows = (uint64_t)(num_blocks * page_block);
  // Q: the 32-dim RoPE halves (64-B swizzle). KV, 16-bit caches: 64-dim latent
  // chunks (128-B swizzle) and 32-dim RoPE halves (64-B swizzle). KV, FP8 rows
  // (bytes): 256 e4m3 per CTA, the 16 scale bytes, 64 RoPE bytes (64-B swizzle).
  // V4.1 rows (bytes): this CTA's data bytes (256 e4m3 or 128 of e2m1 pairs)
  // and 16 scale bytes; their queries are read by the kernel without a map.
  CUtensorMap tm_qr, tm_kv, tm_kvr, tm_sc;
  const bool few_heads = h_q == kFewHeads;
  if (few_heads) {
    // few heads: Q of one query position as one box of all 9 chunks of 64
    // dims; a 64-token tile as four boxes of two latent chunks and one of the
    // RoPE chunk
    if (!make_map_chunks(&tm_qr, q, dt, (uint64_t)qrows, kFewHeads, 9) ||
        !make_map_chunks(&tm_kv, kvcache, dt, kvrows, 64, 2) || !make_map_chunks(&tm_kvr, kvcache, dt, kvrows, 64, 1))
      return MLA_ERR_CUDA;
    tm_sc = tm_kv;
  } else if (!v41 && !make_map(&tm_qr, q, dt, 2, (uint64_t)qrows, kDK, kDK * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B)) {
    return MLA_ERR_CUDA;
  }
  if (few_heads) {
  } else if (v41) {
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int rb = kv_format == MLA_KV_FP4_288 ? kRowBytesFp4_288 : kRowBytesFp8_528;
    const int data = kv_format == MLA_KV_FP4_288 ? 128 : 256;
    const int box_rows = sparse ? 1 : 64;  // sparse: TMA gather4, one-row boxes
    if (!make_map(&tm_kv, kvcache, u8, 1, kvrows, rb, rb, data, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_sc, kvcache, u8, 1, kvrows, rb, rb, 16, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MLA_ERR_CUDA;
    tm_qr = tm_kvr = tm_kv;  // not read
  } else if (mode == dense::MODE_FP8_SPARSE) {
    // rows gathered four at a time (TMA gather4: one-row boxes, no swizzle):
    // this CTA's 256 e4m3 bytes, the 16 scale bytes, its 64 RoPE bytes
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map(&tm_kv, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_sc, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 16, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_kvr, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 64, 1, CU_TENSOR_MAP_SWIZZLE_64B))
      return MLA_ERR_CUDA;
  } else if (mode == dense::MODE_FP8) {
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map(&tm_kv, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 256, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_sc, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_kvr, kvcache, u8, 1, kvrows, kRowBytesFp8, kRowBytesFp8, 64, 64, CU_TENSOR_MAP_SWIZZLE_64B))
      return MLA_ERR_CUDA;
  } else {
    if (!make_map_chunks(&tm_kv, kvcache, dt, kvrows, 64, 4) ||
        !make_map(&tm_kvr, kvcache, dt, 2, kvrows, kDK, kDK * 2, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
      return MLA_ERR_CUDA;
    tm_sc = tm_kv;
  }

  const int64_t S = max_splits(batch * s_q, parts);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.q = q;
  p.block_table = block_table;
  p.seqlens = cache_seqlens;
  p.indices = indices;
  p.kv = static_cast<const uint8_t*>(kvcache);
  p.meta = static_cast<const int32_t*>(metadata);
  p.split_off = num_splits;
  p.out = out;
  p.out_v8 = aligned(out, 32) ? 1 : 0;
  p.lse = lse;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.o_part = reinterpret_cast<float*>(ws + kWsHeader);
  p.lse_part = p.o_part + S * h_q * kDV;
  p.exact_flags = reinterpret_cast<uint32_t*>(ws + ws_flags_offset(batch * s_q, parts, h_q));
  p.num_blocks = num_blocks;
  p.num_rows = num_blocks * page_block;
  p.max_blocks = max_blocks;
  p.batch = batch;
  p.s_q = s_q;
  p.h_q = h_q;
  p.topk = topk;
  p.causal = causal ? 1 : 0;
  p.kv_format = kv_format;
  p.parts = parts;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.stall_cycles = g_test_stall.load(std::memory_order_relaxed);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the decode kernels wait for the preceding grid themselves (griddepcontrol),
  // so they are launched as programmatic dependents of it
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if ((stages & STAGE_SPLIT) && few_heads) {
    cudaLaunchConfig_t cfg = {};
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(parts, 1, 1);
    cfg.blockDim = dim3(few::kThreads, 1, 1);
    cfg.dynamicSmemBytes = few::kSmemBytes;
    cfg.stream = st;
    if (fp16)
      MLA_CUDA(cudaLaunchKernelEx(&cfg, few::mla_decode_fewheads_kernel<true>, tm_qr, tm_kv, tm_kvr, p));
    else
      MLA_CUDA(cudaLaunchKernelEx(&cfg, few::mla_decode_fewheads_kernel<false>, tm_qr, tm_kv, tm_kvr, p));
  } else if (stages & STAGE_SPLIT) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * parts, 1, 1);
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cfg.stream = st;
    MLA_CUDA(launch_decode_mode(mode, cfg, tm_qr, tm_kv, tm_kvr, tm_sc, p));
  }
  if (!(stages & STAGE_COMBINE)) return MLA_OK;

  // combine, overlapped with the decode grid's tail (programmatic dependent launch)
  CombineParams c{num_splits, p.o_part, p.lse_part, out, lse, batch, s_q, h_q, fp16 ? 1 : 0};
  if (kv_format == MLA_KV_16BIT && !indices && h_q == 128) {  // the kernels that flag rows for an exact recompute
    c.exact_flags = p.exact_flags;
    c.q = q;
    c.kv = p.kv;
    c.block_table = block_table;
    c.seqlens = cache_seqlens;
    c.num_blocks = num_blocks;
    c.max_blocks = max_blocks;
    c.causal = causal ? 1 : 0;
    c.scale_log2 = p.scale_log2;
  }
  cudaLaunchConfig_t cc = {};
  // 16 heads: 8 blocks per request share its 64 output units (no row is
  // flagged for an exact recompute there, which every block would repeat)
  const bool z8 = c.exact_flags == nullptr && h_q <= 16;
  cc.gridDim = dim3(batch * s_q, (h_q + 15) / 16, z8 ? 8 : 1);
  cc.blockDim = dim3(256, 1, 1);
  cc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cc.attrs = at;
  cc.numAttrs = 1;
  if (fp16 && z8)
    MLA_CUDA(cudaLaunchKernelEx(&cc, mla_combine_kernel<__half, 1>, c));
  else if (fp16)
    MLA_CUDA(cudaLaunchKernelEx(&cc, mla_combine_kernel<__half, 8>, c));
  else if (z8)
    MLA_CUDA(cudaLaunchKernelEx(&cc, mla_combine_kernel<__nv_bfloat16, 1>, c));
  else
    MLA_CUDA(cudaLaunchKernelEx(&cc, mla_combine_kernel<__nv_bfloat16, 8>, c));
  return MLA_OK;
}
}  // namespace

extern "C" {

#define MLA_DECODE_ARGS                                                                                        \
  q, q_dtype, kvcache, num_blocks, page_block, block_table, max_blocks, cache_seqlens, batch, s_q, h_q,         \
      head_dim_v, metadata, num_splits, parts, softmax_scale, causal, kv_format, indices, topk, out, lse, workspace, \
      workspace_bytes, stream
#define MLA_DECODE_PARAMS                                                                                         \
  const void *q, int q_dtype, const void *kvcache, int64_t num_blocks, int page_block, const int32_t *block_table, \
      int max_blocks, const int32_t *cache_seqlens, int batch, int s_q, int h_q, int head_dim_v,                   \
      const void *metadata, const int32_t *num_splits, int parts, float softmax_scale, int causal, int kv_format,     \
      const int32_t *indices, int topk, void *out, float *lse, void *workspace, size_t workspace_bytes,            \
      void *stream

mla_status mla_decode_with_kvcache(MLA_DECODE_PARAMS) {
  return decode_impl(STAGE_SPLIT | STAGE_COMBINE, MLA_DECODE_ARGS);
}
mla_status mla_decode_splitkv(MLA_DECODE_PARAMS) { return decode_impl(STAGE_SPLIT, MLA_DECODE_ARGS); }
mla_status mla_combine_splits(MLA_DECODE_PARAMS) { return decode_impl(STAGE_COMBINE, MLA_DECODE_ARGS); }

mla_status mla_quantize_kv_fp8(const void* kv, uint8_t* out, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!kv || !out))) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  int dev = 0, sms = 0;
  MLA_CUDA(cudaGetDevice(&dev));
  MLA_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t want = (n + 7) / 8;
  const int grid = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  mla_quant_fp8_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint16_t*>(kv), out, n);
  MLA_CUDA(cudaGetLastError());
  return MLA_OK;
}

static mla_status quantize_v41(const void* kv, uint8_t* out, int64_t n, bool fp4, void* stream) {
  if (n < 0 || (n > 0 && (!kv || !out))) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  int dev = 0, sms = 0;
  MLA_CUDA(cudaGetDevice(&dev));
  MLA_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t want = (n + 7) / 8;  // one warp per row, 8 warps per block
  const int grid = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  const uint16_t* src = static_cast<const uint16_t*>(kv);
  if (fp4)
    mla_quant_fp4_288_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(src, out, n);
  else
    mla_quant_fp8_528_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(src, out, n);
  MLA_CUDA(cudaGetLastError());
  return MLA_OK;
}

mla_status mla_quantize_kv_fp8_528(const void* kv, uint8_t* out, int64_t n, void* stream) {
  return quantize_v41(kv, out, n, false, stream);
}

mla_status mla_quantize_kv_fp4_288(const void* kv, uint8_t* out, int64_t n, void* stream) {
  return quantize_v41(kv, out, n, true, stream);
}

mla_status mla_absorb_q(const void* q_nope, const void* w_uk, void* q_out, int tokens, int h_q, int dtype,
                        uint32_t* status, void* stream) {
  if (tokens < 0 || h_q < 1 || (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_FP16)) return MLA_ERR_INVALID_ARG;
  if (status && !aligned(status, 4)) return MLA_ERR_INVALID_ARG;
  if (tokens == 0) return MLA_OK;
  if (!q_nope || !w_uk || !q_out || !aligned(q_nope, 16) || !aligned(w_uk, 16) || !aligned(q_out, 16))
    return MLA_ERR_INVALID_ARG;
  const CUtensorMapDataType dt =
      dtype == MLA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t H = (cuuint64_t)h_q, T = (cuuint64_t)tokens;
  // q_nope [T, h, 128] as {64 dims, tokens, 2 chunks, heads}: tiles [chunk][token][64]
  CUtensorMap tm_a, tm_b;
  if (!make_map_4d(&tm_a, q_nope, dt, {64, T, 2, H}, {H * 256, 128, 256}, {64, absorb::kTokTile, 2, 1}) ||
      // w_uk [h, 128, 512] as {64 latent dims, 128 rows, 8 chunks, heads}: [chunk][row][64]
      !make_map_4d(&tm_b, w_uk, dt, {64, 128, 8, H}, {1024, 128, 128 * 1024}, {64, 128, 8, 1}))
    return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t stall = g_test_stall.load(std::memory_order_relaxed);
  const dim3 grid((unsigned)h_q, (unsigned)((tokens + absorb::kTokTile - 1) / absorb::kTokTile));
  if (dtype == MLA_DTYPE_FP16) {
    MLA_CUDA(set_smem(absorb::mla_absorb_q_kernel<true>, absorb::kAbsorbSmem));
    absorb::mla_absorb_q_kernel<true><<<grid, absorb::kThreads, absorb::kAbsorbSmem, st>>>(tm_a, tm_b, q_out, tokens,
                                                                                           h_q, status, stall);
  } else {
    MLA_CUDA(set_smem(absorb::mla_absorb_q_kernel<false>, absorb::kAbsorbSmem));
    absorb::mla_absorb_q_kernel<false><<<grid, absorb::kThreads, absorb::kAbsorbSmem, st>>>(tm_a, tm_b, q_out, tokens,
                                                                                            h_q, status, stall);
  }
  MLA_CUDA(cudaGetLastError());
  return MLA_OK;
}

mla_status mla_up_project(const void* o_lat, const void* w_uv, void* o_out, int tokens, int h_q, int dtype,
                          uint32_t* status, void* stream) {
  if (tokens < 0 || h_q < 1 || (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_FP16)) return MLA_ERR_INVALID_ARG;
  if (status && !aligned(status, 4)) return MLA_ERR_INVALID_ARG;
  if (tokens == 0) return MLA_OK;
  if (!o_lat || !w_uv || !o_out || !aligned(o_lat, 16) || !aligned(w_uv, 16) || !aligned(o_out, 16))
    return MLA_ERR_INVALID_ARG;
  const CUtensorMapDataType dt =
      dtype == MLA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t H = (cuuint64_t)h_q, T = (cuuint64_t)tokens;
  // o_lat [T, h, 512] as {64 dims, tokens, 8 chunks, heads}: tiles [chunk][token][64]
  CUtensorMap tm_a, tm_b;
  if (!make_map_4d(&tm_a, o_lat, dt, {64, T, 8, H}, {H * 1024, 128, 1024}, {64, absorb::kTokTile, 4, 1}) ||
      // w_uv [h, 128, 512] as {64 latent dims, 128 rows, 8 chunks, heads}: [chunk][row][64]
      !make_map_4d(&tm_b, w_uv, dt, {64, 128, 8, H}, {1024, 128, 128 * 1024}, {64, 128, 4, 1}))
    return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t stall = g_test_stall.load(std::memory_order_relaxed);
  const dim3 grid((unsigned)h_q, (unsigned)((tokens + absorb::kTokTile - 1) / absorb::kTokTile));
  if (dtype == MLA_DTYPE_FP16) {
    MLA_CUDA(set_smem(absorb::mla_up_project_kernel<true>, absorb::kUpSmem));
    absorb::mla_up_project_kernel<true><<<grid, absorb::kThreads, absorb::kUpSmem, st>>>(tm_a, tm_b, o_out, tokens,
                                                                                         h_q, status, stall);
  } else {
    MLA_CUDA(set_smem(absorb::mla_up_project_kernel<false>, absorb::kUpSmem));
    absorb::mla_up_project_kernel<false><<<grid, absorb::kThreads, absorb::kUpSmem, st>>>(tm_a, tm_b, o_out, tokens,
                                                                                          h_q, status, stall);
  }
  MLA_CUDA(cudaGetLastError());
  return MLA_OK;
}

mla_status mla_read_status(void* workspace, void* stream, uint32_t* bits) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  MLA_CUDA(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st));
  MLA_CUDA(cudaStreamSynchronize(st));
  MLA_CUDA(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st));
  MLA_CUDA(cudaStreamSynchronize(st));
  if (bits) *bits = v;
  if (v & STATUS_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (v & STATUS_STALE) return MLA_ERR_STALE_METADATA;
  if (v & STATUS_INDEX) return MLA_ERR_INDEX;
  if (v & STATUS_RANGE) return MLA_ERR_RANGE;
  return MLA_OK;
}

void mla_set_test_stall(uint32_t cycles) { g_test_stall.store(cycles, std::memory_order_relaxed); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of mla_decode_with_kvcache.
//
// Some callers cannot obtain device memory on demand: cudaMalloc may
// synchronise the whole device and can fail once memory is committed, which a
// serving loop with a fixed latency budget, or a plug-in running inside a host
// application that owns every device allocation, cannot accept. For them the
// split-KV scratch (the status word and the fp32 partial outputs of cut
// requests) lives in one fixed device array compiled into this library. Every
// GPU that loads the library holds its own copy of the array until the
// process exits, and all calls on one device share that copy: calls that
// overlap on the GPU (for example on two streams) race on it and must be
// serialised by the caller.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kStaticWsBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

std::mutex g_static_mu[kMaxDevices];
std::atomic<void*> g_static_ptr[kMaxDevices];

// Host code may not use g_static_ws directly (its name is a host-side stand-in,
// not a device address): look the device address up with that device current,
// and keep it once the lookup has succeeded. A failed lookup (for example one
// made during a stream capture) is not remembered: the next call tries again.
void* static_ws_ptr(int dev, cudaError_t* err) {
  *err = cudaSuccess;
  void* ptr = g_static_ptr[dev].load(std::memory_order_acquire);
  if (ptr) return ptr;
  std::lock_guard<std::mutex> lock(g_static_mu[dev]);
  ptr = g_static_ptr[dev].load(std::memory_order_relaxed);
  if (ptr) return ptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_ws);
  if (e != cudaSuccess || !ptr) {
    (void)cudaGetLastError();
    *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    return nullptr;
  }
  g_static_ptr[dev].store(ptr, std::memory_order_release);
  return ptr;
}
}  // namespace

extern "C" mla_status mla_decode_with_kvcache_noalloc(
    const void* q, int q_dtype, const void* kvcache, int64_t num_blocks, int page_block, const int32_t* block_table,
    int max_blocks, const int32_t* cache_seqlens, int batch, int s_q, int h_q, int head_dim_v, const void* metadata,
    const int32_t* num_splits, int parts, float softmax_scale, int causal, int kv_format, const int32_t* indices, int topk,
    void* out, float* lse, uint32_t* status, void* stream) {
  const size_t need = mla_workspace_size(batch, s_q, h_q, parts);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > kStaticWsBytes) return MLA_ERR_INVALID_ARG;  // beyond the fixed scratch: use mla_decode_with_kvcache
  if (status && !aligned(status, 4)) return MLA_ERR_INVALID_ARG;
  // every argument check happens before the first enqueue (the status
  // memset); the fixed array is the workspace, sized and aligned above
  const mla_status v = validate_decode(q, q_dtype, kvcache, num_blocks, page_block, block_table, max_blocks,
                                       cache_seqlens, batch, s_q, h_q, head_dim_v, metadata, num_splits, parts,
                                       softmax_scale, causal, kv_format, indices, topk, out, lse, false, nullptr, 0);
  if (v != MLA_OK) return v;
  int dev = 0;
  MLA_CUDA(cudaGetDevice(&dev));
  if (dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  cudaError_t e = cudaSuccess;
  void* ws = static_ws_ptr(dev, &e);
  if (e != cudaSuccess || !ws) return MLA_ERR_CUDA;
  // The array keeps the previous call's contents: the status word must start
  // at zero (the fp32 partials are fully written before they are read).
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MLA_CUDA(cudaMemsetAsync(ws, 0, sizeof(uint32_t), st));
  mla_status r = decode_impl(STAGE_SPLIT | STAGE_COMBINE, q, q_dtype, kvcache, num_blocks, page_block, block_table,
                             max_blocks, cache_seqlens, batch, s_q, h_q, head_dim_v, metadata, num_splits, parts,
                             softmax_scale, causal, kv_format, indices, topk, out, lse, ws, kStaticWsBytes, stream);
  // device-side problems (bad index or page, stale metadata, wait timeout) are
  // recorded in the array's status word; copy them out for the caller
  if (r == MLA_OK && status) MLA_CUDA(cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st));
  return r;
}
