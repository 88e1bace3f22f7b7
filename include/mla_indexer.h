/*
 * mla_indexer.h -- C ABI of the GB300 (sm_103a) Lightning Indexer + top-k.
 *
 * Operation ("CANN DeepSeek Indexer attention", sections "Lightning Indexer"
 * and "Sparse Flash Attention"): for every query token t = (b, s) and every
 * candidate key position j of its sequence,
 *
 *     I[t, j] = sum_h w[t, h] * ReLU(q[t, h, :] . k[row(b, j), :])
 *
 * and the token attends to Top-k(I[t, :]), which this call returns as the
 * topk_idx input of mla_sparse_attn_fwd (mla_sparse.h).
 *
 *   candidates     j in [0, act_seqs[b]); row(b, j) = block_table[b, j / 128] *
 *                  128 + j % 128 (the same paging as the attention cache).  A
 *                  position whose block id lies outside [0, num_blocks) (or
 *                  whose table slot is beyond max_blocks_per_seq) is not a
 *                  candidate and raises MLA_DEVICE_BAD_BLOCK.
 *   selection      the min(topk, #candidates) largest scores; among equal
 *                  scores the smaller position wins, so the result is unique.
 *   output order   ascending positions, then -1 up to topk.
 *
 * Conventions are those of mla_sparse.h: device pointers owned by the caller,
 * asynchronous on `stream`, argument errors returned before any launch with
 * mla_indexer_last_error() describing them, every internal wait bounded
 * (mla_sparse_set_wait_limit_ns); a wait that runs out makes that launch give
 * up and raises MLA_DEVICE_TIMEOUT, and the next launch runs in full.
 * Numerics: q and k bf16, products exact, dot products and the head sum in
 * fp32 (tensor cores, fp32 accumulate); the selection compares those fp32
 * scores exactly.
 */
#ifndef MLA_INDEXER_H_
#define MLA_INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#include "mla_sparse.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_indexer_dims {
  int32_t B;                  /* sequences */
  int32_t S1;                 /* query tokens per sequence */
  int32_t n_heads;            /* indexer heads H: a multiple of 16, S1 * H <= 256 */
  int32_t head_dim;           /* D: 128 */
  int32_t block_size;         /* 128 */
  int32_t num_blocks;         /* physical blocks in k_cache */
  int32_t max_blocks_per_seq; /* block_table row width W */
  int32_t topk;               /* >= 1 */
} mla_indexer_dims;

/* Bytes of workspace mla_indexer_topk needs: B * S1 * W * 128 fp32 scores.
 * Returns 0 for invalid dims. */
size_t mla_indexer_workspace_bytes(const mla_indexer_dims* dims);

/*
 * q           bf16 [B*S1, H, D]
 * w           fp32 [B*S1, H]           head weights of each token
 * k_cache     bf16 [num_blocks*128, D] the paged index-key cache (16-byte aligned)
 * block_table int32 [B, W]
 * act_seqs    int32 [B]
 * topk_idx    int32 [B*S1, topk]       output
 * workspace   device memory of at least mla_indexer_workspace_bytes(dims),
 *             256-byte aligned, owned by the caller; on return it holds the
 *             scores as fp32 [B*S1, W*128]: entry [t, j] = I[t, j] for
 *             candidate positions j, -inf for positions below act_seqs[b] that
 *             are not candidates, unspecified at and beyond act_seqs[b].
 * Two launches on `stream` (mla_indexer_scores into the workspace, then
 * mla_indexer_select as a programmatic dependent launch, so its launch
 * overlaps the score grid's tail).  MLA_ERR_SHAPE when the workspace is too
 * small.
 */
mla_status mla_indexer_topk(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                            const int32_t* block_table, const int32_t* act_seqs, int32_t* topk_idx,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two phases of mla_indexer_topk as separate calls (one launch each), for
 * callers that want the scores themselves or select from scores of their own.
 *
 * mla_indexer_scores: the score phase alone.  scores is the fp32 [B*S1, W*128]
 * buffer of at least mla_indexer_workspace_bytes(dims) bytes, 256-byte
 * aligned, filled as the workspace of mla_indexer_topk is.
 */
mla_status mla_indexer_scores(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                              const int32_t* block_table, const int32_t* act_seqs, float* scores,
                              size_t scores_bytes, void* stream);

/*
 * mla_indexer_select: the selection phase alone, on any fp32 scores laid out
 * as above (row t = b*S1 + s, leading dimension W*128): among positions
 * j < act_seqs[b], -inf marks a non-candidate and every other value must be
 * finite; entries at and beyond act_seqs[b] are not read.  dims->q-side
 * fields (n_heads, head_dim, num_blocks) are checked as for the score phase.
 */
mla_status mla_indexer_select(const mla_indexer_dims* dims, const float* scores, const int32_t* act_seqs,
                              int32_t* topk_idx, void* stream);

/*
 * mla_indexer_topk_noalloc: mla_indexer_topk without a workspace argument.
 * No counterpart in the method as described ("CANN DeepSeek Indexer
 * attention"); it serves callers that cannot allocate device memory at call
 * time, such as a host program that sizes all its device memory once at
 * start-up, where a later cudaMalloc could fail or wait for the whole device.
 *
 * The scores go to a scratch array inside the library's device image (8 MiB,
 * created by the CUDA runtime with the module): the call allocates nothing.
 *   limit       B * S1 * max_blocks_per_seq * 128 <= 2,097,152 scores; larger
 *               dims return MLA_ERR_SHAPE before any launch, with a message.
 *   races       one scratch per device and process: calls that overlap in time
 *               (on other streams or from other host threads) overwrite each
 *               other's scores.  Serialise them, or use mla_indexer_topk.
 *   first call  the first call on each device looks the scratch address up
 *               (cudaGetSymbolAddress) and keeps it; make that first call
 *               before any stream capture begins.
 *   zeroing     none is needed: every score the selection reads is written
 *               by the score phase of the same call.
 * Arguments, outputs, launches and errors are otherwise those of
 * mla_indexer_topk.
 */
mla_status mla_indexer_topk_noalloc(const mla_indexer_dims* dims, const void* q, const float* w,
                                    const void* k_cache, const int32_t* block_table, const int32_t* act_seqs,
                                    int32_t* topk_idx, void* stream);

/* Description of the last error of an mla_indexer_* call on this thread
 * (empty after a successful call). */
const char* mla_indexer_last_error(void);

/* Synchronises `stream`, returns the indexer's sticky device status bits
 * (MLA_DEVICE_BAD_BLOCK, MLA_DEVICE_TIMEOUT) and clears them when `clear` is
 * nonzero; MLA_ERR_DEVICE_STATUS when any bit is set. */
mla_status mla_indexer_device_status(void* stream, uint32_t* flags, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* MLA_INDEXER_H_ */
