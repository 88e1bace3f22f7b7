/*
 * mla_prolog.h -- C ABI of the GB300 (sm_103a) MLA Prolog: hidden states to
 * the absorbed query of mla_sparse_attn_fwd (mla_sparse.h) plus the new key
 * row written into its paged cache.
 *
 * Operation ("NPU DeepSeek-V4 PyPTO fused-operator optimization", section
 * MlaProlog, both formula groups; "CANN DeepSeek Indexer attention", section
 * MLA Prolog: the DeepSeek-V3 structure with weight absorption in decode, and
 * the fused prototype's weights w_dq, w_uq_qr, w_uk, w_dkv_kr, gamma_cq,
 * gamma_ckv, sin, cos, cache_index), for every token t:
 *
 *   c^Q      = RMSNorm(x[t] @ wq_a) * gamma_cq                 (q_lora wide)
 *   q[h]     = RMSNorm((c^Q @ wq_b)[h])                        (per head, 192 wide, weight 1)
 *   q_rope   = RoPE(q[h][128:192])                             -> q_rope[t, h]
 *   q_nope   = q[h][0:128] @ w_uk[h]                           -> q_nope[t, h] (512 wide)
 *   k        = RMSNorm(x[t] @ wkv) * gamma_ckv                 (576 wide, one norm over the row)
 *   the cache row cache_index[t] receives k[0:512] and RoPE(k[512:576]).
 *
 *   RMSNorm(v) = v / sqrt(mean(v^2) + eps).
 *   RoPE       interleaved pairs (2i, 2i+1), i < 32:
 *              y[2i] = v[2i] cos[t,i] - v[2i+1] sin[t,i],
 *              y[2i+1] = v[2i] sin[t,i] + v[2i+1] cos[t,i].
 *   cache      written exactly as mla_cache_write (mla_cache.h) writes the
 *              bf16 row k: negative index skipped, index >= num_rows skipped
 *              and MLA_DEVICE_BAD_BLOCK raised, INT8 by 128-element groups.
 *
 * Numerics: the matrix products run on tensor cores with bf16 operands and
 * fp32 accumulation; c^Q and q[h][0:128] are stored as bf16 (they are the
 * next products' operands); norms and rotations are fp32; q_nope, q_rope and
 * the cache row are rounded to bf16 once, at the end.
 *
 * Conventions are those of mla_sparse.h: device pointers owned by the caller,
 * asynchronous on `stream`, argument errors returned before any launch with
 * mla_prolog_last_error() describing them.  Every step runs in this
 * library's kernels: the four matrix products in its tcgen05 product kernel
 * (the weights streamed by TMA as the MMA's A operand, x @ wq_a and x @ wkv
 * in one launch), the norms, rotations and the cache write in its row
 * kernels; all five launches go to `stream`, so the call is capturable into a
 * CUDA graph.  The first call on each device sets the product kernel's
 * shared-memory attribute and looks up the driver's tensor-map encoder: make
 * it before any stream capture begins.
 */
#ifndef MLA_PROLOG_H_
#define MLA_PROLOG_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_sparse.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_prolog_dims {
  int32_t T;         /* tokens, >= 0 (0: no-op) */
  int32_t hidden;    /* model width, a positive multiple of 8 */
  int32_t q_lora;    /* query latent width, a positive multiple of 8 */
  int32_t n_heads;   /* query heads H >= 1; T * H < 2^31 */
  int64_t num_rows;  /* cache rows (num_blocks * block_size) >= 1 */
  int32_t kv_int8;   /* 0: bf16 cache, 1: INT8 cache with fp32 group scales */
  float eps;         /* RMSNorm epsilon, > 0 */
} mla_prolog_dims;

typedef struct mla_prolog_weights {
  const void* wq_a;      /* bf16 [hidden, q_lora]              (row-major, x @ wq_a) */
  const void* gamma_cq;  /* bf16 [q_lora] */
  const void* wq_b;      /* bf16 [q_lora, H * 192]; head h owns columns [192 h, 192 h + 192),
                            its first 128 without position, its last 64 rotated */
  const void* w_uk;      /* bf16 [H, 128, 512]                 (absorption) */
  const void* wkv;       /* bf16 [hidden, 576]; columns [0, 512) latent, [512, 576) rope */
  const void* gamma_ckv; /* bf16 [576] */
} mla_prolog_weights;

/* Bytes of workspace mla_prolog needs (the fp32 partial sums of the
 * projections over their k splits and the bf16 operands between the
 * products); 0 for invalid dims. */
size_t mla_prolog_workspace_bytes(const mla_prolog_dims* dims);

/*
 * x           bf16 [T, hidden]
 * w           the weights above (the struct itself is read on the host)
 * cos, sin    fp32 [T, 32]      one rotation per rope pair
 * cache_index int64 [T]
 * q_nope      bf16 [T, H, 512]  output
 * q_rope      bf16 [T, H, 64]   output
 * kv_nope     [num_rows, 512]   bf16 or int8, updated in place
 * kv_rope     bf16 [num_rows, 64], updated in place
 * kv_scales   fp32 [num_rows, 4] (INT8 only; NULL for bf16), updated in place
 * workspace   >= mla_prolog_workspace_bytes(dims) bytes, 256-byte aligned
 * Every pointer 16-byte aligned (cache_index 8-byte).  Five launches on
 * `stream` (the two x projections, the c^Q and key rows, c^Q @ wq_b, the
 * per-head norms, the absorption), each a programmatic dependent of the
 * previous one; MLA_ERR_SHAPE when the workspace is too small.
 */
mla_status mla_prolog(const mla_prolog_dims* dims, const void* x, const mla_prolog_weights* w, const float* cos,
                      const float* sin, const int64_t* cache_index, void* q_nope, void* q_rope, void* kv_nope,
                      void* kv_rope, float* kv_scales, void* workspace, size_t workspace_bytes, void* stream);

/* Description of the last error of an mla_prolog* call on this thread. */
const char* mla_prolog_last_error(void);

/* Synchronises `stream`, returns the prolog's sticky device status bits
 * (MLA_DEVICE_BAD_BLOCK) and clears them when `clear` is nonzero;
 * MLA_ERR_DEVICE_STATUS when any bit is set. */
mla_status mla_prolog_device_status(void* stream, uint32_t* flags, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* MLA_PROLOG_H_ */
