/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) decode over a
 * paged, compressed latent KV cache, for NVIDIA GB300 (sm_103a).
 *
 * What is computed. After weight absorption every query head scores one shared
 * 576-wide cache row per token (512 latent dims c^KV + 64 decoupled-RoPE dims
 * k^R): score = q~ . c + q^R . k^R, and the value is the 512-wide latent c
 * itself; decode is therefore MQA with h_kv = 1, d_k = 576, d_v = 512
 * ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §六 '吸收' and '结果：decode
 * 变成 MQA'). For every request b, query position i and head h:
 *     out[b,i,h,:] = sum_t softmax_t(scale * q[b,i,h,:] . K_t) * K_t[0:512]
 *     lse[b,i,h]   = ln sum_t exp(scale * q[b,i,h,:] . K_t)
 * over the visible tokens t (§五 '注意力：两个 GEMM 加一个 softmax' of the same
 * page; the kernels use the online softmax and the split-KV combine of §五/§七,
 * which reorder but do not approximate it).
 *
 * Conventions for every call below:
 *  - Pointers marked (device) are CUDA device pointers owned by the caller; the
 *    library never allocates, frees or retains them past the call (except that
 *    the kernels it enqueues read/write them until they complete on `stream`).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued asynchronously; no call synchronises the host except
 *    mla_read_status().
 *  - Argument errors are detected on the host before anything is enqueued and
 *    return MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED; nothing is written then.
 *  - Problems only visible on the device (an out-of-range page or index, a
 *    stale metadata buffer, a pipeline wait that timed out) never trap: the
 *    kernel sets a bit in the status word kept in the workspace, and
 *    mla_read_status() reports it.
 *  - All entry points are thread-safe; calls on one stream execute in order.
 */
#ifndef MLA_GB300_H_
#define MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,      /* bad shape, pointer, alignment or flag combination */
  MLA_ERR_UNSUPPORTED = 2,      /* valid request the library does not implement   */
  MLA_ERR_STALE_METADATA = 3,   /* metadata computed for a different shape/lengths */
  MLA_ERR_INDEX = 4,            /* an out-of-range page or sparse index was skipped */
  MLA_ERR_TIMEOUT = 5,          /* a device pipeline wait gave up (kernel returned early) */
  MLA_ERR_CUDA = 6,             /* a CUDA runtime/driver call failed */
  MLA_ERR_RANGE = 7             /* quantised cache: a value or a score beyond the certified range (see below) */
} mla_status;

typedef enum { MLA_DTYPE_BF16 = 0, MLA_DTYPE_FP16 = 1 } mla_dtype;

/* Cache row formats (the `kv_format` argument; 0 and 1 are the reference's
 * is_fp8_kvcache = false / true):
 *  MLA_KV_16BIT    576 values of q_dtype (512 latent + 64 RoPE), 1152 B;
 *  MLA_KV_FP8_656  512 e4m3 latent values, 4 fp32 scales (one per 128), the 64
 *                  RoPE dims as bf16: 656 B ("FlashMLA 实战：MLA 注意力加速指南",
 *                  §FP8 缓存怎么把 KV 压掉四成);
 *  MLA_KV_FP8_528  the V4.1 row of 512 values (latent and RoPE together): 512
 *                  e4m3 codes, then 16 UE8M0 scales, byte j = k + 127 for the
 *                  scale 2^k of values [32j, 32j+32): 528 B;
 *  MLA_KV_FP4_288  the FP4 row of 512 values: 256 bytes of e2m1 codes (value 2i
 *                  in the low nibble of byte i), then 32 e4m3 scales, byte j for
 *                  values [16j, 16j+16): 288 B
 * ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA", §八 '版本漂移' and the §十
 * format table). With the V4.1 rows a key is 512 wide and the value is the
 * whole row: q is [batch, s_q, h_q, 512] and head_dim_v is 512. */
typedef enum { MLA_KV_16BIT = 0, MLA_KV_FP8_656 = 1, MLA_KV_FP8_528 = 2, MLA_KV_FP4_288 = 3 } mla_kv_format;

#define MLA_HEAD_DIM_K 576
#define MLA_HEAD_DIM_V 512
#define MLA_FP8_ROW_BYTES 656
#define MLA_V41_DIM 512
#define MLA_FP8_528_ROW_BYTES 528
#define MLA_FP4_288_ROW_BYTES 288

/* Human-readable name of a status code (static string). */
MLA_API const char* mla_status_string(int status);

/* Number of work partitions ("SM parts") the 128-head decode kernels use on
 * `device`: the number of co-resident 2-CTA clusters of the dense/FP8 decode
 * kernel. Returns a value <= 0 on failure (no device). */
MLA_API int mla_num_sm_parts(int device);

/* The same for a given number of query heads: h_q = 128 as above; h_q = 16
 * (the transposed few-heads kernel, one CTA per part, after the FlashMLA-ETAP
 * page, §3.1) the number of its co-resident CTAs. Returns a value <= 0 on
 * failure or for an unsupported h_q. */
MLA_API int mla_num_sm_parts_for(int device, int h_q);

/* Bytes of the metadata buffer for a decode shape. */
MLA_API size_t mla_metadata_size(int batch, int s_q, int num_sm_parts);

/*
 * Split-KV work schedule ("矩阵、注意力与 GPU：拆解 DeepGEMM 与 FlashMLA",
 * §七 'split-KV：把长序列切开': the schedule decides which SM part handles which
 * requests and KV blocks and how many pieces each request is cut into; it is
 * computed once and reused by every layer and step of the same shape).
 *
 * The (request, query position) pairs v = i*batch + b ("virtual requests")
 * are cut into 64-token tiles (visible length per query position: dense
 * L_b, or L_b - s_q + 1 + i when causal; sparse: topk) and the tile list is
 * cut into `num_sm_parts` contiguous ranges of nearly equal cost.
 *
 * cache_seqlens (device) int32 [batch]; may be NULL when topk > 0 (sparse).
 * metadata      (device) mla_metadata_size() bytes, written.
 * num_splits    (device) int32 [batch*s_q + 1], written: exclusive prefix sum
 *               of the number of pieces of each virtual request.
 * kv_format: an mla_kv_format, the one the decode calls will pass.
 * h_q must be 128, or 16 for dense 16-bit caches (the few-heads kernel);
 * h_kv must be 1, page_block 64.
 * Computed entirely on the device (no host synchronisation). The decode call
 * checks on the device that the metadata matches its own arguments and the
 * current cache_seqlens, and reports MLA_ERR_STALE_METADATA otherwise.
 */
MLA_API mla_status mla_get_metadata(const int32_t* cache_seqlens, int batch, int s_q, int h_q, int h_kv,
                            int topk, int kv_format, int causal, int page_block, int num_sm_parts,
                            void* metadata, int32_t* num_splits, void* stream);

/* Bytes of decode workspace (status word, fp32 split partials, and one bit per
 * (query position, head) row for the exact recompute). */
MLA_API size_t mla_workspace_size(int batch, int s_q, int h_q, int num_sm_parts);

/*
 * Decode attention over the latent cache ("FlashMLA 实战：MLA 注意力加速指南",
 * §最小调用: out, lse = flash_mla_with_kvcache(q, kvcache, block_table,
 * cache_seqlens, head_dim_v=512, metadata, num_splits, softmax_scale, causal,
 * is_fp8_kvcache, indices)).
 *
 * q            (device) [batch, s_q, h_q, 576] (V4.1 rows: 512), `q_dtype`,
 *              contiguous, 16-B aligned; bf16 with every quantised format.
 * kvcache      (device) [num_blocks, page_block, 1, row] contiguous, 16-B
 *              aligned: 576 values of q_dtype (kv_format = MLA_KV_16BIT), or
 *              uint8 rows of 656, 528 or 288 bytes (MLA_KV_FP8_656,
 *              MLA_KV_FP8_528, MLA_KV_FP4_288; see the quantisers below).
 *              Token-sparse decode (indices) reads the quantised formats.
 * block_table  (device) int32 [batch, max_blocks], logical page -> physical page;
 *              may be NULL when indices != NULL.
 * cache_seqlens(device) int32 [batch] tokens per request (ignored when indices != NULL).
 * head_dim_v   must be 512.
 * metadata, num_splits: from mla_get_metadata() with the same shape/flags.
 * softmax_scale: multiplies q.K (e.g. 576^-0.5).
 * causal       bottom-right aligned mask for s_q > 1; must be 0 with indices.
 * indices      (device) int32 [batch, s_q, topk] absolute cache rows
 *              (page * page_block + slot), -1 = unused slot; NULL for dense.
 *              Rows must lie in [0, num_blocks*page_block); others are skipped
 *              and flagged as MLA_ERR_INDEX ("拆解" page, §八 sparse indices).
 * out          (device) [batch, s_q, h_q, 512] of q_dtype, written.
 * lse          (device) fp32 [batch, s_q, h_q], natural log, written.
 * workspace    (device) mla_workspace_size() bytes, 256-B aligned, zeroed once
 *              before first use: it holds the status word (mla_read_status
 *              clears it), the fp32 partials of cut requests and one bit per
 *              (query position, head) row that the combine recomputes exactly
 *              (the library leaves those bits zero after every call).
 * A request with no visible token gets out = 0 and lse = -inf.
 * 656-byte FP8 rows run the latent product in fp16: the bf16 query is
 * rounded to fp16 and each cache value is formed as fp16(code) x fp16(block
 * scale), rounded to fp16. Within range the dequantised value has relative
 * error <= 2^-10; a block whose amax is below 448 * 2^-14 (~0.027) has an
 * fp16-subnormal scale, and its values carry an absolute error <= 2^-15
 * instead. Out of range -- a query entry beyond 65504 in magnitude (saturated
 * to +-65504) or a block scale above 146 (block amax above 65408) -- the
 * status word records MLA_ERR_RANGE.
 * The V4.1 rows run in fp16 as well (query rounded to fp16, with the same
 * 65504 limit): e2m1 x e4m3 is always exact in fp16; e4m3 x 2^k is exact for
 * k in [-15, 7]; a block with a smaller scale (amax below 448 * 2^-16) carries
 * an absolute error of at most 2^-25, and a larger one (amax above 57344,
 * UE8M0 byte above 134) is reported as MLA_ERR_RANGE.
 * Every cache type splits the dims of a score between the two CTAs of a
 * pair, which exchange fp16 factors 2^(partial score - partial max). The
 * result is certified exact (to fp16 precision) for a row of a 64-token tile
 * unless the two partial scores of its tokens disagree by more than about 22
 * binades; such a row is recomputed exactly from q and the cache rows for
 * 16-bit caches (by the combine step, so mla_decode_splitkv alone leaves it
 * uncorrected until mla_combine_splits runs), and reported as MLA_ERR_RANGE
 * for quantised caches.
 * h_q = 128 with any cache; h_q = 16 with a dense 16-bit cache only: the few
 * heads fill the MMA's N dimension and the 64 tokens of a tile its M
 * dimension, the transposed formulation S^T = K Q^T, O^T = V^T P^T of the
 * FlashMLA-ETAP page (§2.2, §3.2); same results and layouts.
 */
MLA_API mla_status mla_decode_with_kvcache(const void* q, int q_dtype, const void* kvcache, int64_t num_blocks,
                                   int page_block, const int32_t* block_table, int max_blocks,
                                   const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                                   int head_dim_v, const void* metadata, const int32_t* num_splits,
                                   int num_sm_parts, float softmax_scale, int causal, int kv_format,
                                   const int32_t* indices, int topk, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two launches mla_decode_with_kvcache() is made of, for callers that
 * schedule them separately (same arguments, same checks):
 *  - mla_decode_splitkv: the split-KV kernel ("矩阵、注意力与 GPU：拆解 DeepGEMM 与
 *    FlashMLA", §七 'split-KV'); requests that are one piece get their final
 *    out/lse, the pieces of cut requests get fp32 partials (o, lse) in the
 *    workspace;
 *  - mla_combine_splits: merges those partials into out/lse (m = max lse_i,
 *    o = sum o_i e^{lse_i - m} / sum e^{lse_i - m}, same section) and writes
 *    out = 0, lse = -inf for requests with no visible token. It must follow
 *    mla_decode_splitkv of the same arguments on the same stream.
 */
MLA_API mla_status mla_decode_splitkv(const void* q, int q_dtype, const void* kvcache, int64_t num_blocks,
                                      int page_block, const int32_t* block_table, int max_blocks,
                                      const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                                      int head_dim_v, const void* metadata, const int32_t* num_splits,
                                      int num_sm_parts, float softmax_scale, int causal, int kv_format,
                                      const int32_t* indices, int topk, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream);
MLA_API mla_status mla_combine_splits(const void* q, int q_dtype, const void* kvcache, int64_t num_blocks,
                                      int page_block, const int32_t* block_table, int max_blocks,
                                      const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                                      int head_dim_v, const void* metadata, const int32_t* num_splits,
                                      int num_sm_parts, float softmax_scale, int causal, int kv_format,
                                      const int32_t* indices, int topk, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_with_kvcache without a caller-supplied workspace, for callers that
 * cannot allocate device memory on demand (cudaMalloc may synchronise the
 * device and can fail once memory is committed -- unacceptable inside a
 * fixed-latency serving loop, or for a plug-in whose host application owns
 * every device allocation). The pages describe no such entry point; it is an
 * engineering addition of this library.
 *
 * Same arguments and results as mla_decode_with_kvcache, except:
 *  - the split-KV scratch is a fixed 32 MiB array inside the library, one per
 *    device, held until the process exits; a shape whose mla_workspace_size()
 *    exceeds 32 MiB is rejected with MLA_ERR_INVALID_ARG (use
 *    mla_decode_with_kvcache for it);
 *  - nothing is allocated or freed;
 *  - all calls on a device share the array: calls that may overlap on the GPU
 *    (e.g. on different streams) race and must be serialised by the caller;
 *  - the first call on a device looks up the array's device address (once,
 *    with that device current); make that first call before any stream
 *    capture;
 *  - status (device, optional, 4-B aligned): receives the device-side status
 *    bits of this call (1 = index/page skipped, 2 = wait timeout, 4 = stale
 *    metadata, 8 = range of a quantised cache), or NULL to discard them.
 */
MLA_API mla_status mla_decode_with_kvcache_noalloc(const void* q, int q_dtype, const void* kvcache,
                                                   int64_t num_blocks, int page_block,
                                                   const int32_t* block_table, int max_blocks,
                                                   const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                                                   int head_dim_v, const void* metadata,
                                                   const int32_t* num_splits, int num_sm_parts,
                                                   float softmax_scale, int causal, int kv_format,
                                                   const int32_t* indices, int topk, void* out, float* lse,
                                                   uint32_t* status, void* stream);

/*
 * Write the 656-byte FP8 cache rows ("FlashMLA 实战：MLA 注意力加速指南",
 * §FP8 缓存怎么把 KV 压掉四成): bytes [0,512) e4m3 codes of the 512 latent dims,
 * quantised per 128 values with scale = fp32(amax/448) (1.0 for an all-zero
 * block) and code = round-to-nearest-even(fp32(x/scale)) saturated to +-448;
 * bytes [512,528) the 4 scales as fp32; bytes [528,656) the 64 RoPE dims copied
 * as bf16.
 * kv (device) bf16 [n, 576] (row stride 576 elements); out (device) uint8 [n, 656].
 */
MLA_API mla_status mla_quantize_kv_fp8(const void* kv, uint8_t* out, int64_t n, void* stream);

/*
 * Write the V4.1 rows of 512 values ("矩阵、注意力与 GPU：拆解 DeepGEMM 与
 * FlashMLA", §八 '版本漂移', §十 format table; §三 'UE8M0': a power-of-two
 * scale, rounded up). The page prints no quantiser; these follow the plainest
 * reading of it, and the oracle defines the same decisions independently:
 *  - mla_quantize_kv_fp8_528: per 32 values the scale is the smallest 2^k
 *    (k >= -127) with 448 * 2^k >= amax; byte 512 + j = k + 127; byte d =
 *    e4m3 round-to-nearest-even of x_d / 2^k (exact division);
 *  - mla_quantize_kv_fp4_288: per 16 values the scale is the smallest
 *    non-negative e4m3 value v with 6 v >= amax (448 when none is, values then
 *    saturate to +-6); byte 256 + j = its code; each value becomes the e2m1
 *    code nearest to x / v (ties to the even code, the sign of x kept), value
 *    2i in the low nibble of byte i.
 * kv (device) bf16 [n, 512] (row stride 512 elements, finite values); out
 * (device) uint8 [n, 528] or [n, 288]; both 16-B aligned.
 */
MLA_API mla_status mla_quantize_kv_fp8_528(const void* kv, uint8_t* out, int64_t n, void* stream);
MLA_API mla_status mla_quantize_kv_fp4_288(const void* kv, uint8_t* out, int64_t n, void* stream);

/*
 * The per-head GEMMs around the kernel ("矩阵、注意力与 GPU：拆解 DeepGEMM 与
 * FlashMLA", §六 '吸收'): with the key up-projection W^UK_i (d_h x d_c) absorbed
 * into the query, q~_{t,i} = W^UK_i^T q^C_{t,i}, every head scores the shared
 * latent row; the value up-projection is applied once to the attention-weighted
 * latent, o_{t,i} = W^UV_i o~_{t,i}. Here d_h = 128 and d_c = 512; tokens is the
 * number of query tokens (batch * s_q), h_q the number of heads; dtype is
 * MLA_DTYPE_BF16 or MLA_DTYPE_FP16 for every operand. Products accumulate in
 * fp32 and are rounded once to dtype. All pointers are (device), 16-B aligned.
 *
 * mla_absorb_q: q_nope [tokens, h_q, 128], w_uk [h_q, 128, 512] (W^UK_i row d
 * holds the 512 latent weights of output dim d); writes dims [0, 512) of every
 * row of q_out [tokens, h_q, 576], the layout mla_decode_with_kvcache reads,
 * and leaves the 64 RoPE dims [512, 576) to the caller.
 *
 * mla_up_project: o_lat [tokens, h_q, 512] (the decode output), w_uv
 * [h_q, 128, 512]; writes o_out [tokens, h_q, 128].
 *
 * status (device, optional, 4-B aligned): a status word the kernels OR bit 2
 * (wait timeout) into when a bounded wait gave up (nothing is stored then);
 * read and clear it with mla_read_status(). NULL discards it.
 *
 * tokens = 0 enqueues nothing. Returns MLA_ERR_INVALID_ARG for a negative size,
 * a null or misaligned pointer, or an unknown dtype.
 */
MLA_API mla_status mla_absorb_q(const void* q_nope, const void* w_uk, void* q_out, int tokens, int h_q, int dtype,
                                uint32_t* status, void* stream);
MLA_API mla_status mla_up_project(const void* o_lat, const void* w_uv, void* o_out, int tokens, int h_q, int dtype,
                                  uint32_t* status, void* stream);

/*
 * Synchronise `stream`, read and clear the status word of `workspace` (or of
 * any 4-B status word, e.g. the one given to mla_absorb_q), and return the
 * first error it records, in the order timeout, stale metadata, index, range
 * (MLA_OK if none). *bits (optional) receives the raw bits: 1 = index/page
 * skipped, 2 = wait timeout, 4 = stale metadata, 8 = range of a quantised cache.
 */
MLA_API mla_status mla_read_status(void* workspace, void* stream, uint32_t* bits);

/*
 * Test hook for the time-out path (0, the default, turns it off). While it is
 * non-zero, every decode kernel (mla_decode_with_kvcache and its variants)
 * and absorption kernel (mla_absorb_q, mla_up_project) launched by this
 * library first has one thread per CTA wait `cycles` SM cycles on a barrier
 * that nothing arrives at, before any copy or MMA is issued; the wait gives up, the kernel records the wait
 * time-out (status bit 2, MLA_ERR_TIMEOUT) and the CTA skips its work, so the
 * outputs of those launches are undefined. Process-wide; not for production
 * use. The pages describe no such hook: it exists so that a test can check that
 * a device wait which runs out is reported and leaves the context usable.
 */
MLA_API void mla_set_test_stall(uint32_t cycles);

#ifdef __cplusplus
}
#endif
#endif /* MLA_GB300_H_ */
