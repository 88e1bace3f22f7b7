/*
 * mla_sparse.h -- C ABI of the GB300 (sm_103a) sparse MLA attention library.
 *
 * Operation (sparse_flash_attention_quant, "DeepSeek V3/V2 Sparse Flash
 * Attention with Quantization": sections "Algorithm overview", "Operator
 * spec", "Inputs / outputs", "Compute pipeline" and "INT8 quantization path";
 * the selection rule is o_i = Attn(x_i, {c_j : j in Top-k(I_i,:)}) from "CANN
 * DeepSeek Indexer attention", section "Sparse Flash Attention"):
 *
 *   for every query token t = (b, s) and query head h (all heads share the one
 *   latent KV head, N_KV = 1):
 *     valid entries  i : 0 <= topk_idx[t, i] < act_seqs[b]
 *     row            r_i = block_table[b, j / 128] * 128 + j % 128, j = topk_idx[t, i]
 *     score          z_i = softmax_scale * (q_nope[t,h,:] . kv_nope[r_i,:]
 *                                         + q_rope[t,h,:] . kv_rope[r_i,:])
 *     out[t,h,:]   = sum_i softmax(z)_i * kv_nope[r_i,:]      (value = key_nope)
 *     lse[t,h]     = ln sum_i exp(z_i)
 *   INT8 cache rows are dequantised per 128-element group as
 *   bf16(fp32(q8) * scale) before use.  A token with no valid entry gets
 *   out = 0 and lse = -inf.  Repeated indices count once per occurrence.
 *
 * Conventions
 *   - Every data pointer is a DEVICE pointer owned by the caller.  Besides a
 *     device status word and the bound of its device-side waits, the library
 *     keeps one buffer per (device, stream) for calls with few tokens and long
 *     lists (whole tokens per cluster would leave the longest cluster at least
 *     twice an equal share of the key tiles): such a call gives every cluster
 *     an equal share, a token cut between clusters leaves one partial softmax
 *     state per part in the buffer, and a second launch merges them.  The
 *     buffer (~40 MB on a GB300) is allocated by the first such call on the
 *     stream and kept for the life of the process (mla_sparse_allow_cut_tokens(0)
 *     turns this off: whole tokens, no buffer).  A first such call on a
 *     stream that is capturing a CUDA graph allocates nothing and schedules
 *     whole tokens instead (same results, less even load).  Calls on one
 *     stream share its buffer in stream order; a captured graph uses the
 *     buffer of the stream it was captured on and must not run concurrently
 *     with other calls on that stream.
 *   - All tensors are dense row-major with the shapes given below.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and never synchronise.
 *   - Argument errors are detected on the host before any launch and return a
 *     negative status; mla_sparse_last_error() then describes the problem
 *     (thread-local, valid until the next call on the same thread).
 *   - Bad block ids for valid indices (outside [0, num_blocks), or a table
 *     slot index / 128 beyond max_blocks_per_seq) never fault: the entry is
 *     masked out of the softmax and MLA_DEVICE_BAD_BLOCK is raised in the
 *     device status word.  Every internal wait of the kernel is bounded (500 ms
 *     unless mla_sparse_set_wait_limit_ns says otherwise); a wait that runs
 *     out makes that launch give up (its out/lse are then unspecified) and
 *     raises MLA_DEVICE_TIMEOUT.  Status bits accumulate until cleared; a
 *     later launch still runs in full.
 *   - Numerics: inputs bf16; products are exact; score and output
 *     accumulation in fp32 on the tensor cores (each CTA of a two-CTA
 *     cluster owns half of the latent and rope dims; the two exchange fp32
 *     partial scores, so both hold the same score tile); a token cut
 *     between clusters is merged in fp32 with the flash update's weights
 *     2^(m_k - max m); the softmax weights P enter
 *     the P.V product as two bf16 terms, P_hi = bf16(p) and
 *     P_lo = bf16(p - P_hi), so their relative error stays below 2^-18; the
 *     values are the bf16 cache rows themselves; out is rounded to bf16 once.
 */
#ifndef MLA_SPARSE_H_
#define MLA_SPARSE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_NULL = -1,           /* a required pointer is NULL */
  MLA_ERR_SHAPE = -2,          /* a dimension is out of range */
  MLA_ERR_DTYPE = -3,          /* kv_dtype unknown, or scales missing for INT8 */
  MLA_ERR_UNSUPPORTED = -4,    /* a valid but unimplemented configuration */
  MLA_ERR_ALIGN = -5,          /* a pointer is not aligned as required */
  MLA_ERR_CUDA = -6,           /* the CUDA runtime reported an error */
  MLA_ERR_DEVICE_STATUS = -7   /* the device status word holds an error */
} mla_status;

typedef enum mla_mode {
  MLA_MODE_DECODE = 0,   /* "Decode mode": standard softmax over the token's selection */
  MLA_MODE_PREFILL = 1   /* "Prefill mode": flash online softmax across key tiles */
} mla_mode;

typedef enum mla_kv_dtype {
  MLA_KV_BF16 = 0,   /* kv_nope holds bf16 */
  MLA_KV_INT8 = 1    /* kv_nope holds int8 with one fp32 scale per 128 elements */
} mla_kv_dtype;

/* Device status bits (mla_sparse_device_status). */
#define MLA_DEVICE_BAD_BLOCK 0x1u
#define MLA_DEVICE_TIMEOUT 0x2u

/*
 * Problem dimensions ("Inputs / outputs" table).  Supported today:
 * n_kv == 1, d_nope == 512 (kv_lora_rank), d_rope == 64 (qk_rope_dim),
 * block_size == 128, 1 <= n_q <= 128, topk >= 1, num_blocks in [1, 2^24).
 */
typedef struct mla_dims {
  int32_t B;                  /* batch */
  int32_t S1;                 /* query tokens per batch entry */
  int32_t n_q;                /* query heads N_Q */
  int32_t n_kv;               /* latent KV heads N_KV */
  int32_t d_nope;             /* kv_lora_rank */
  int32_t d_rope;             /* qk_rope_dim */
  int32_t block_size;         /* paged-cache block size */
  int32_t num_blocks;         /* physical blocks in the cache */
  int32_t max_blocks_per_seq; /* width of block_table */
  int32_t topk;               /* entries per token in topk_idx */
  int32_t kv_dtype;           /* mla_kv_dtype */
} mla_dims;

/*
 * mla_sparse_attn_fwd -- sparse MLA attention forward over a paged cache.
 *
 *   q_nope      bf16 [B*S1, n_q, d_nope]                       16-byte aligned
 *   q_rope      bf16 [B*S1, n_q, d_rope]                       16-byte aligned
 *   kv_nope     bf16 | int8 [num_blocks*block_size, d_nope]    16-byte aligned
 *   kv_rope     bf16 [num_blocks*block_size, d_rope]           16-byte aligned
 *   kv_scales   fp32 [num_blocks*block_size, d_nope/128]; required (16-byte
 *               aligned) for MLA_KV_INT8, ignored for MLA_KV_BF16
 *   topk_idx    int32 [B*S1, n_kv*topk]: logical positions; entries < 0 or
 *               >= act_seqs[b] are masked
 *   block_table int32 [B, max_blocks_per_seq]: physical block of each logical block
 *   act_seqs    int32 [B]: actual KV length of each batch entry
 *   out         bf16 [B, S1, n_q, d_nope] (written)                16-byte aligned
 *               (32-byte aligned: stored 32 bytes per instruction, faster)
 *   lse         fp32 [B, S1, n_q] (written) or NULL
 *   softmax_scale  finite scale applied to the summed nope + rope score
 *   mode        mla_mode: selects the schedule only; both modes compute the
 *               same function
 *   stream      cudaStream_t
 *
 * Returns MLA_OK once the work is enqueued, or a negative mla_status.
 */
mla_status mla_sparse_attn_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope,
                               const void* kv_nope, const void* kv_rope, const float* kv_scales,
                               const int32_t* topk_idx, const int32_t* block_table,
                               const int32_t* act_seqs, void* out, float* lse, float softmax_scale,
                               int32_t mode, void* stream);

/*
 * mla_swa_fwd -- sliding-window attention over the same paged cache ("NPU
 * DeepSeek-V4 PyPTO fused-operator optimization", section SWA: attention over
 * the original KV with a sliding-window mask, for prefill and MTP).  The S1
 * query tokens of sequence b are its newest S1 positions: token (b, s) sits at
 * p = act_seqs[b] - S1 + s and attends to the positions [p - window + 1, p]
 * that are >= 0.  The pages give no window size: `window` (>= 1) is the
 * caller's.  Arguments as mla_sparse_attn_fwd without topk_idx; dims->topk is
 * ignored.  Same kernel, with each token's position list built on the device
 * instead of read.
 */
mla_status mla_swa_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope, const void* kv_nope,
                       const void* kv_rope, const float* kv_scales, const int32_t* block_table,
                       const int32_t* act_seqs, int32_t window, void* out, float* lse, float softmax_scale,
                       int32_t mode, void* stream);

/*
 * mla_compressed_attn_fwd -- compressed and sparse compressed flash attention
 * (CFA / SCFA, "NPU DeepSeek-V4 PyPTO fused-operator optimization", sections
 * CFA, SCFA and Compressor): each query token attends, under one softmax, to
 * its window of the original cache and to entries of a compressed cache.
 *   token (b, s) sits at p = act_seqs[b] - S1 + s; original part: positions
 *   [p - window + 1, p] that are >= 0 (as mla_swa_fwd);
 *   compressed entry i (the Compressor's output for positions
 *   [i*ratio, (i+1)*ratio)) is visible iff (i+1)*ratio - 1 <= p;
 *   CFA (sparse_idx == NULL): every visible entry; SCFA: the visible entries
 *   of sparse_idx[b*S1 + s, 0:topk] (logical entry ids; others masked).
 * The compressed cache has the original cache's row layout and dtype
 * (dims->kv_dtype; INT8 rows need scales), paged by its own block table.
 * Arguments otherwise as mla_swa_fwd; dims->topk is ignored.  Rows of either
 * cache must stay below 2^30 (num_blocks < 2^23).
 */
typedef struct mla_cmp_cache {
  const void* nope;           /* [num_blocks*128, d_nope] bf16 | int8, 16-byte aligned */
  const void* rope;           /* [num_blocks*128, d_rope] bf16, 16-byte aligned */
  const float* scales;        /* [num_blocks*128, d_nope/128] for INT8, else NULL */
  const int32_t* block_table; /* [B, max_blocks_per_seq] */
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t ratio;              /* compress ratio r >= 1 */
  const int32_t* sparse_idx;  /* NULL (CFA) or [B*S1, topk] int32 (SCFA) */
  int32_t topk;               /* width of sparse_idx (SCFA), ignored for CFA */
} mla_cmp_cache;

mla_status mla_compressed_attn_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope,
                                   const void* kv_nope, const void* kv_rope, const float* kv_scales,
                                   const int32_t* block_table, const mla_cmp_cache* cmp,
                                   const int32_t* act_seqs, int32_t window, void* out, float* lse,
                                   float softmax_scale, int32_t mode, void* stream);

/* Description of the last error on this thread ("" after a success). */
const char* mla_sparse_last_error(void);

/*
 * Synchronises `stream`, reads the device status word of the current device
 * into *flags (MLA_DEVICE_* bits; flags may be NULL) and clears it when
 * `clear` is non-zero.  Returns MLA_ERR_DEVICE_STATUS if any bit was set,
 * MLA_ERR_CUDA on a runtime error, MLA_OK otherwise.
 */
mla_status mla_sparse_device_status(void* stream, uint32_t* flags, int32_t clear);

/*
 * mla_sparse_get_device_status -- the status query under the name of the
 * boundary's original list: mla_sparse_device_status(stream, NULL, 0), i.e.
 * synchronise, report without clearing.
 */
mla_status mla_sparse_get_device_status(void* stream);

/*
 * mla_sparse_set_wait_limit_ns -- bound, in nanoseconds, of every device-side
 * wait of the library's launches enqueued after this call: the attention
 * kernels, the Lightning Indexer's score kernel and the MLA Prolog's product
 * kernel (all threads of the process; default 500 ms).  Waits that only let
 * copies or MMAs already in flight land before a block exits keep at least
 * 500 ms.  No counterpart in the pages: the pages' runtime
 * debug mode ("DeepSeek V3/V2 Sparse Flash Attention with Quantization",
 * notes) checks the operator while it runs; this bound is what turns a stall
 * into MLA_DEVICE_TIMEOUT instead of a hang.  Accepted range [1 us, 60 s];
 * MLA_ERR_SHAPE otherwise.  A short bound makes a launch whose waits take
 * longer give up, which the tests use to exercise the timeout path.
 */
mla_status mla_sparse_set_wait_limit_ns(uint64_t ns);

/*
 * mla_sparse_launch_count -- number of kernel launches the attention entry
 * points (mla_sparse_attn_fwd, mla_swa_fwd, mla_compressed_attn_fwd) have
 * enqueued in this process so far, all threads and devices together.  One per
 * call, two when a call cuts tokens between clusters (the attention kernel
 * and the merge of the cut tokens' parts).  For accounting only.
 */
uint64_t mla_sparse_launch_count(void);

/*
 * mla_sparse_allow_cut_tokens -- whether later attention calls may give the
 * persistent clusters equal shares of the key tiles, cutting tokens between
 * them (allow != 0, the default), or always schedule whole tokens (0).  With
 * 0 the library never allocates its buffer for cut tokens and every call is a
 * single launch; results are the same either way, only the load balance of
 * calls with few tokens and long lists differs.  Applies to all threads of
 * the process.
 */
void mla_sparse_allow_cut_tokens(int32_t allow);

/* ABI version of this header (major * 100 + minor). */
int32_t mla_sparse_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_SPARSE_H_ */
