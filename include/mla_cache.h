/*
 * mla_cache.h -- C ABI of the GB300 (sm_103a) paged MLA cache writer.
 *
 * Operation: write T new key rows into the paged cache that
 * mla_sparse_attn_fwd (mla_sparse.h) reads.  The cache layout is the one of
 * "DeepSeek V3/V2 Sparse Flash Attention with Quantization" (sections on the
 * operator spec and inputs/outputs): key_nope_2d (rows, 512) BF16 or INT8,
 * key_rope_2d (rows, 64) BF16, k_nope_scales (rows, 4) FP32 with one scale
 * per 128 elements; the INT8 rule is the page's quantisation note (groups of
 * 128, absolute maximum as the scale, values into [-128, 127]).  The writer
 * is the cache-update step of the MlaProlog operator ("NPU DeepSeek-V4 PyPTO
 * fused-operator optimization", section MlaProlog, cache_index).
 *
 *   cache_index[t]  the flat physical row (block id * block_size + offset) of
 *                   new row t; negative: no row (skipped); at or beyond
 *                   num_rows: skipped, and MLA_DEVICE_BAD_BLOCK is raised.
 *                   Indices are expected to be distinct (with duplicates the
 *                   row that lands is unspecified).
 *   bf16 cache      the nope and rope rows are copied bit for bit.
 *   INT8 cache      per 128-element group g: scale = absmax / 127 in fp32 (1
 *                   when that is not positive), code = clamp(round half to
 *                   even (x / scale), -128, 127) with the division in fp32;
 *                   kv_scales[row, g] = scale.  The rope row is copied.
 *
 * Conventions are those of mla_sparse.h: device pointers owned by the caller,
 * asynchronous on `stream` (one launch), argument errors returned before any
 * launch with mla_cache_last_error() describing them.
 */
#ifndef MLA_CACHE_H_
#define MLA_CACHE_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_sparse.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * k_nope      bf16 [T, 512]     new latent rows
 * k_rope      bf16 [T, 64]      new rope rows
 * cache_index int64 [T]
 * kv_nope     [num_rows, 512]   bf16 (kv_int8 = 0) or int8 (kv_int8 = 1), updated in place
 * kv_rope     bf16 [num_rows, 64], updated in place
 * kv_scales   fp32 [num_rows, 4] (INT8 only; NULL for bf16), updated in place
 * All 16-byte aligned (cache_index 8-byte).  T = 0 is a no-op that reads no
 * pointer (they may be NULL).
 */
mla_status mla_cache_write(int32_t T, int64_t num_rows, int32_t kv_int8, const void* k_nope, const void* k_rope,
                           const int64_t* cache_index, void* kv_nope, void* kv_rope, float* kv_scales,
                           void* stream);

/* Description of the last error of an mla_cache_* call on this thread. */
const char* mla_cache_last_error(void);

/* Synchronises `stream`, returns the writer's sticky device status bits
 * (MLA_DEVICE_BAD_BLOCK) and clears them when `clear` is nonzero;
 * MLA_ERR_DEVICE_STATUS when any bit is set. */
mla_status mla_cache_device_status(void* stream, uint32_t* flags, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* MLA_CACHE_H_ */
