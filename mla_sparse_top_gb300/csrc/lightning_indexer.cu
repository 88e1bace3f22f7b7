// Lightning Indexer + top-k for GB300 (sm_103a).
//
// "CANN DeepSeek Indexer attention", section "Lightning Indexer": the index
// score of query token t for key position j is
//     I[t, j] = sum_h w[t, h] * ReLU(q[t, h, :] . k[j, :]),
// and (section "Sparse Flash Attention") the token attends to Top-k(I[t, :]).
//
// Kernel 1 (scores).  The keys of a sequence are consecutive positions, so a
// 128-key tile is exactly one cache block: 128 contiguous rows of 256 bytes,
// fetched by two TMA tiled loads (64 dims each, 128-byte swizzle).  The
// S1 * H query rows of a sequence (its tokens x indexer heads, N <= 256) stay
// in shared memory.  One tcgen05 MMA chain per tile computes
//     D[key, (token, head)] = K_tile . Q^T      (M = 128 keys, N, K = 128 dims)
// into TMEM, so each epilogue thread owns one key (one TMEM lane) and the
// weighted ReLU sum over heads is thread-local.  TMEM holds up to four
// accumulators, so the MMAs of the next tiles overlap the epilogue of tile i.
//   warp 0      TMA producer (one thread), key ring of up to 6 stages
//   warp 1      TMEM allocation and MMA issue (one thread)
//   warps 2-3   load the sequence's head weights once (its Q rows come by TMA,
//               issued by the producer ahead of the first key tile)
//   warps 4-11  epilogue, two warpgroups that split the tokens (a warp reads
//               TMEM lanes 32 * (warp % 4) ...): ReLU, weights, head sum,
//               fp32 scores to the workspace
//
// Kernel 2 (selection), one CTA per token: an exact select on the
// order-preserving 32-bit image of the fp32 scores finds the k-th largest key T
// and how many entries equal to T are kept (a value-bucket histogram narrows
// the search to one bucket, whose keys are then ranked directly; byte-wise
// radix passes cover the cases bucketing cannot); a compaction in position
// order then writes the positions with key > T and the first ones with
// key == T, so the output is ascending and ties go to the smaller position.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/mla_indexer.h"
#include "ptx.cuh"

namespace mlasp {
unsigned long long host_wait_limit_ns();  // the library's wait bound (mla_sparse_set_wait_limit_ns)
}

namespace mlaidx {
using namespace mlasp;

constexpr int kBlock = 128;                  // keys per tile = rows per cache block
constexpr int kDim = 128;                    // head_dim
constexpr int kMaxStages = 6;               // key-tile ring depth: as many 32 KB stages as fit
constexpr int kChunkBytes = kBlock * 128;    // 128 rows x 64 bf16 dims (128-byte swizzled rows)
constexpr int kTileBytes = 2 * kChunkBytes;  // 32 KB
constexpr int kMaxN = 256;                   // S1 * H
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiGroups = 2;                // epilogue warpgroups; group g takes tokens g, g + 2, ...
constexpr int kEpiThreads = 128 * kEpiGroups;
constexpr int kMaxAcc = 4;                   // TMEM accumulators (tiles in flight between MMA and epilogue)

// Shared memory: the small items first, then the sequence's Q rows (two
// 64-dim chunks of N rows), then the key ring; the last two are placed at run
// time from N (qchunk = N * 128 bytes, stages = what fits, <= kMaxStages).
constexpr int kOffW = 0;                     // N fp32 head weights
constexpr int kOffBars = kOffW + kMaxN * 4;
constexpr int kBarFull = 0;                  // [kMaxStages]
constexpr int kBarEmpty = kBarFull + kMaxStages;  // [kMaxStages]
constexpr int kBarTFull = kBarEmpty + kMaxStages;  // [kMaxAcc]
constexpr int kBarTEmpty = kBarTFull + kMaxAcc;  // [kMaxAcc]
constexpr int kBarQReady = kBarTEmpty + kMaxAcc;
constexpr int kBarFinal = kBarQReady + 1;    // the MMA thread's last commit
constexpr int kNumBars = kBarFinal + 1;
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffQ = 2048;
constexpr int kSmemMax = 232448;             // 227 KB, the per-block opt-in limit
static_assert(kOffAbort + 4 <= kOffQ, "small items fit below Q");
static_assert(kOffQ % 1024 == 0 && kTileBytes % 1024 == 0, "operand alignment");
static_assert(kOffQ + 2 * kMaxN * 128 + 2 * kTileBytes <= kSmemMax, "at least two stages at the largest N");

// Waits that only let copies or MMAs already in flight land before the CTA
// exits are never cut shorter than this, whatever the configured bound.
constexpr uint64_t kDrainWaitNs = 500ull * 1000ull * 1000ull;

__device__ unsigned int g_idx_status = 0;

struct ScoreParams {
  const uint16_t* q;
  const float* w;
  const int32_t* block_table;
  const int32_t* act_seqs;
  float* scores;
  int64_t ld;  // scores row stride (floats)
  int S1, H, N, num_blocks, mbps, tiles_per_cta;
  int n_acc;  // TMEM accumulators of N columns each, <= kMaxAcc
  int stages;  // key-ring depth, <= kMaxStages
  uint32_t q_chunk;     // bytes of one 64-dim chunk of Q: N * 128
  uint32_t off_stages;  // shared-memory offset of the key ring
  uint32_t tmem_cols;
  unsigned long long wait_ns;  // bound of every wait (mla_sparse_set_wait_limit_ns)
};

struct Ctx {
  uint32_t sbase;
  uint8_t* smem;
  volatile uint32_t* abort;
  uint64_t wait_ns;
  __device__ uint32_t bar(int i) const { return sbase + kOffBars + 8 * i; }
};

__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity) {
  return mbar_wait<false>(c.bar(idx), parity, c.abort, c.wait_ns);
}
__device__ __forceinline__ bool warp_wait(const Ctx& c, int idx, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(c, idx, parity));
}

// sum_h w[h] * ReLU(D[lane, col + h]) over H heads for this thread's key (TMEM
// lane), NC x 16 heads per TMEM wait (H a multiple of 16 * NC), four partial
// sums.  When `release` is set, the accumulator barrier is arrived on as soon
// as the last columns are in registers, before their arithmetic.
template <int NC>
__device__ __forceinline__ float head_sum(uint32_t col, const float* ws, int H, bool release, uint32_t empty_bar) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int h0 = 0; h0 < H; h0 += 16 * NC) {
    uint32_t v[16 * NC];
#pragma unroll
    for (int k = 0; k < NC; ++k)
      tmem_ld_32x32b_x16(col + static_cast<uint32_t>(h0 + 16 * k), *reinterpret_cast<uint32_t(*)[16]>(&v[16 * k]));
    tmem_wait_ld();
    if (release && h0 + 16 * NC >= H) {
      tc_fence_before();
      mbar_arrive(empty_bar);
    }
    const float4* w4 = reinterpret_cast<const float4*>(ws + h0);
#pragma unroll
    for (int e = 0; e < 16 * NC; e += 4) {
      const float4 ww = w4[e >> 2];
      a0 = fmaf(ww.x, fmaxf(__uint_as_float(v[e + 0]), 0.f), a0);
      a1 = fmaf(ww.y, fmaxf(__uint_as_float(v[e + 1]), 0.f), a1);
      a2 = fmaf(ww.z, fmaxf(__uint_as_float(v[e + 2]), 0.f), a2);
      a3 = fmaf(ww.w, fmaxf(__uint_as_float(v[e + 3]), 0.f), a3);
    }
  }
  return (a0 + a1) + (a2 + a3);
}

__global__ void __launch_bounds__(kThreads, 1)
idx_scores_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ ScoreParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int act = __ldg(p.act_seqs + b);
  const int n_tiles = min((max(act, 0) + kBlock - 1) / kBlock, p.mbps);
  const int tile0 = blockIdx.x * p.tiles_per_cta;
  const int ntile = min(p.tiles_per_cta, n_tiles - tile0);
  if (ntile <= 0) return;  // uniform: this CTA has no key tile

  Ctx c;
  c.smem = smem;
  c.sbase = smem_u32(smem);
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
  c.wait_ns = p.wait_ns;
  if (tid == 0) {
    // each launch starts afresh: a timeout of an earlier launch stays in the
    // status word until it is cleared but does not stop this one
    const bool misaligned = (c.sbase & 1023u) != 0;
    *c.abort = misaligned ? 1u : 0u;
    if (misaligned) atomicOr(&g_idx_status, MLA_DEVICE_TIMEOUT);
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(c.bar(kBarFull + i), 1);
      mbar_init(c.bar(kBarEmpty + i), 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(c.bar(kBarTFull + i), 1);
      mbar_init(c.bar(kBarTEmpty + i), kEpiThreads);
    }
    mbar_init(c.bar(kBarQReady), 1 + 64);  // the producer (Q bytes) and the 64 weight loaders
    mbar_init(c.bar(kBarFinal), 1);
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(c.sbase + kOffTmemSlot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
  // a selection grid launched behind this one may be scheduled now; it waits
  // for this grid's completion before it reads any score
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t qrow0 = static_cast<int64_t>(b) * p.N;  // the sequence's (token, head) rows are contiguous

  if (!*c.abort) {
    if (warp == 0) {
      // ---- TMA producer
      if (lane == 0) {
        // the sequence's N query rows, two 64-dim boxes in the operand's 128-byte swizzled layout
        mbar_arrive_expect_tx(c.bar(kBarQReady), static_cast<uint32_t>(p.N) * kDim * 2);
        tma_load_2d(c.sbase + kOffQ, &qmap, 0, static_cast<int32_t>(qrow0), c.bar(kBarQReady));
        tma_load_2d(c.sbase + kOffQ + p.q_chunk, &qmap, 64, static_cast<int32_t>(qrow0), c.bar(kBarQReady));
        const int32_t* tbl = p.block_table + static_cast<int64_t>(b) * p.mbps + tile0;
        int issued = 0;
        int blk_next = __ldg(tbl);
        for (int i = 0; i < ntile; ++i) {
          const int st = i % p.stages;
          const int blk = blk_next;
          if (i + 1 < ntile) blk_next = __ldg(tbl + i + 1);  // in flight during the wait
          if (!wait_bar(c, kBarEmpty + st, ((i / p.stages) & 1) ^ 1)) break;
          ++issued;
          if (blk >= 0 && blk < p.num_blocks) {
            const uint32_t dst = c.sbase + p.off_stages + st * kTileBytes;
            mbar_arrive_expect_tx(c.bar(kBarFull + st), kTileBytes);
            tma_load_2d(dst, &kmap, 0, blk * kBlock, c.bar(kBarFull + st));
            tma_load_2d(dst + kChunkBytes, &kmap, 64, blk * kBlock, c.bar(kBarFull + st));
          } else {
            // not a candidate block: the epilogue writes -inf for its keys
            atomicOr(&g_idx_status, MLA_DEVICE_BAD_BLOCK);
            mbar_arrive(c.bar(kBarFull + st));
          }
        }
        // every copy issued here lands before the CTA may exit, even after an abort
        volatile uint32_t never = 0;
        mbar_wait<false>(c.bar(kBarQReady), 0, &never, c.wait_ns > kDrainWaitNs ? c.wait_ns : kDrainWaitNs);
        for (int i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i)
          mbar_wait<false>(c.bar(kBarFull + i % p.stages), (i / p.stages) & 1, &never, c.wait_ns > kDrainWaitNs ? c.wait_ns : kDrainWaitNs);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---- MMA issue
      if (lane == 0 && wait_bar(c, kBarQReady, 0)) {
        const uint32_t idesc = make_idesc_f16(128, static_cast<uint32_t>(p.N), 1, 0, 0);
        for (int i = 0; i < ntile; ++i) {
          const int st = i % p.stages, buf = i % p.n_acc;
          if (!wait_bar(c, kBarFull + st, (i / p.stages) & 1)) break;
          if (!wait_bar(c, kBarTEmpty + buf, ((i / p.n_acc) & 1) ^ 1)) break;
          tc_fence_after();
          const uint32_t a0 = c.sbase + p.off_stages + st * kTileBytes;
          const uint32_t b0 = c.sbase + kOffQ;
          const uint32_t d = tmem + static_cast<uint32_t>(buf * p.N);
#pragma unroll
          for (int s = 0; s < 8; ++s)
            umma_ss(d, make_sdesc(a0 + (s >> 2) * kChunkBytes + (s & 3) * 32, 16, 1024, kSwizzle128B),
                    make_sdesc(b0 + (s >> 2) * p.q_chunk + (s & 3) * 32, 16, 1024, kSwizzle128B), idesc,
                    s > 0 ? 1u : 0u);
          umma_commit(c.bar(kBarTFull + buf));
          umma_commit(c.bar(kBarEmpty + st));
        }
      }
      if (lane == 0) {
        // no MMA may still run when TMEM is released, even after an abort
        umma_commit(c.bar(kBarFinal));
        volatile uint32_t never = 0;
        mbar_wait<false>(c.bar(kBarFinal), 0, &never, c.wait_ns > kDrainWaitNs ? c.wait_ns : kDrainWaitNs);
      }
      __syncwarp();
    } else if (warp < kEpiWarp0) {
      // ---- head weights, once
      const int t2 = tid - 64;
      float* wsm = reinterpret_cast<float*>(smem + kOffW);
      for (int n = t2; n < p.N; n += 64) wsm[n] = __ldg(p.w + qrow0 + n);
      mbar_arrive(c.bar(kBarQReady));
    } else {
      // ---- epilogue: thread = key (TMEM lane)
      const int q4 = warp & 3;
      const int eg = (warp - kEpiWarp0) >> 2;
      const int kin = q4 * 32 + lane;
      const float* wsm = reinterpret_cast<const float*>(smem + kOffW);
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const bool have_w = warp_wait(c, kBarQReady, 0);  // the weights are in shared memory
      for (int i = 0; have_w && i < ntile; ++i) {
        const int buf = i % p.n_acc, tl = tile0 + i;
        const int blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.mbps + tl);  // in flight during the wait
        if (!warp_wait(c, kBarTFull + buf, (i / p.n_acc) & 1)) break;
        tc_fence_after();
        const bool valid_blk = blk >= 0 && blk < p.num_blocks;
        const int j = tl * kBlock + kin;
        const uint32_t d = tmem + lane_off + static_cast<uint32_t>(buf * p.N);
        // The accumulator is released as soon as its last columns are in registers,
        // before the arithmetic and the score stores (head_sum of the last token).
        bool released = false;
        for (int s = eg; s < p.S1; s += kEpiGroups) {
          const bool last_token = s + kEpiGroups >= p.S1;
          const float* ws = wsm + s * p.H;
          const uint32_t col = d + static_cast<uint32_t>(s * p.H);
          const float acc = (p.H & 63) == 0 ? head_sum<4>(col, ws, p.H, last_token, c.bar(kBarTEmpty + buf))
                                            : head_sum<1>(col, ws, p.H, last_token, c.bar(kBarTEmpty + buf));
          released |= last_token;
          if (j < act) p.scores[(static_cast<int64_t>(b) * p.S1 + s) * p.ld + j] = valid_blk ? acc : -INFINITY;
        }
        if (!released) {  // a warpgroup without a token of its own
          tc_fence_before();
          mbar_arrive(c.bar(kBarTEmpty + buf));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, p.tmem_cols);
  if (tid == 0 && *c.abort) atomicOr(&g_idx_status, MLA_DEVICE_TIMEOUT);
}

// ------------------------------------------------------------------ selection
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kRegChunks = 8;                        // scores of the first 8192 positions live in registers
constexpr int kSelGroup = kRegChunks * kSelThreads;  // positions per segment
constexpr int kBuckets = 2048;                       // value buckets of the first selection step
constexpr int kListCap = 256;                        // threshold-bucket keys ranked directly
constexpr int kBucketsPerThread = kBuckets / kSelThreads;  // the bucket scan's share of each thread
static_assert(kBucketsPerThread * kSelThreads == kBuckets && kRegChunks * kSelWarps == 256, "selection layout");

struct SelectParams {
  const float* scores;
  int64_t ld;
  int S1;
  const int32_t* act_seqs;
  int32_t* topk_idx;
  int topk;
};

// Order-preserving image of a float: a > b  <=>  key(a) > key(b), and
// a == b  <=>  key(a) == key(b) (no NaN; -0 and +0 share one key).  -inf, which
// marks a position that is not a candidate, would map to 0x007fffff, below
// every finite score; it is treated as key 0 instead.  Every finite score maps
// above 0x007fffff, so keys 0 and 1 never belong to a candidate.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = f == 0.f ? 0u : __float_as_uint(f);
  if (f == -INFINITY) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Value bucket of a candidate score v (vmin <= v <= vmax): a non-decreasing
// function of v, because halving, subtracting a constant, multiplying by a
// positive constant, clamping and truncating are each monotone under
// round-to-nearest; so equal scores share a bucket and every score of a higher
// bucket is larger than every score of a lower one.  Halving keeps vmax - vmin
// finite for any finite pair.  Explicitly rounded operations: no call site may
// contract them differently, since every site must agree on every bucket.
__device__ __forceinline__ int value_bucket(float v, float lo_half, float scale) {
  const float x = __fmul_rn(__fsub_rn(__fmul_rn(v, 0.5f), lo_half), scale);
  return static_cast<int>(fminf(x, static_cast<float>(kBuckets - 1)));
}

// One CTA per token.  Position j = g * 8192 + c * 1024 + tid sits in chunk c of
// segment g; segment 0 keeps its scores in registers, later segments (sequences
// longer than 8192) reload theirs.  The selection keeps every key above a
// threshold key T and the first k_rem keys equal to T, in position order:
//   1. candidate count, min and max (block reduction); all candidates are
//      kept when there are at most topk of them;
//   2. a histogram over kBuckets value buckets and a block scan from the top
//      find the bucket b that holds the topk-th largest score;
//   3. the keys of bucket b (usually a handful) are ranked directly in shared
//      memory, which gives T and k_rem;  when bucketing does not apply (all
//      scores equal, a range too small to scale) or bucket b holds more than
//      kListCap keys, four byte-wise radix passes over the keys of bucket b
//      (of all candidates) do the same;
//   4. compaction in position order.
__global__ void __launch_bounds__(kSelThreads) idx_topk_kernel(const SelectParams p) {
  __shared__ uint32_t hb[kBuckets];  // bucket histogram; radix histograms [2][256] in the fallback
  __shared__ uint32_t cnt[2][kRegChunks * kSelWarps];  // [0] gt / selected, [1] equal; per (chunk, warp)
  __shared__ uint32_t list[kListCap];
  __shared__ float red_lo[kSelWarps], red_hi[kSelWarps];
  __shared__ uint32_t red_n[kSelWarps];
  __shared__ uint32_t bcast[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int t = blockIdx.x;
  const int act = __ldg(p.act_seqs + t / p.S1);
  // positions past the block table's width have no block: not candidates
  if (tid == 0 && static_cast<int64_t>(act) > p.ld) atomicOr(&g_idx_status, MLA_DEVICE_BAD_BLOCK);
  const int n = static_cast<int>(min(static_cast<int64_t>(max(act, 0)), p.ld));
  const int segments = (n + kSelGroup - 1) / kSelGroup;
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  int32_t* out = p.topk_idx + static_cast<int64_t>(t) * p.topk;
  const uint32_t topk = static_cast<uint32_t>(p.topk);

  // When launched behind the score grid (programmatic dependent launch), wait
  // for it to complete and its scores to be visible; otherwise a no-op.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float vreg[kRegChunks];
#pragma unroll
  for (int c = 0; c < kRegChunks; ++c) {
    const int j = c * kSelThreads + tid;
    vreg[c] = j < n ? __ldg(row + j) : -INFINITY;
  }
  auto val_at = [&](int g, int c) -> float {
    if (g == 0) return vreg[c];
    const int j = g * kSelGroup + c * kSelThreads + tid;
    return j < n ? __ldg(row + j) : -INFINITY;
  };
  for (int i = tid; i < kBuckets; i += kSelThreads) hb[i] = 0;
  if (tid < 8) bcast[tid] = 0;

  // ---- 1. candidates, min, max
  {
    uint32_t nc = 0;
    float lo = INFINITY, hi = -INFINITY;
    for (int g = 0; g < segments; ++g) {
#pragma unroll
      for (int c = 0; c < kRegChunks; ++c) {
        const float v = val_at(g, c);
        const bool cand = v != -INFINITY;
        nc += cand ? 1u : 0u;
        lo = cand ? fminf(lo, v) : lo;
        hi = fmaxf(hi, v);
      }
    }
    nc = __reduce_add_sync(0xffffffffu, nc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      red_n[warp] = nc;
      red_lo[warp] = lo;
      red_hi[warp] = hi;
    }
  }
  __syncthreads();
  uint32_t n_cand = 0;
  float vmin = INFINITY, vmax = -INFINITY;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w) {
    n_cand += red_n[w];
    vmin = fminf(vmin, red_lo[w]);
    vmax = fmaxf(vmax, red_hi[w]);
  }

  uint32_t T = 1, k_rem = 0;  // T = 1, k_rem = 0 keeps every candidate (every key > 1)
  if (n_cand > topk) {
    const float lo_half = __fmul_rn(vmin, 0.5f);
    const float range = __fsub_rn(__fmul_rn(vmax, 0.5f), lo_half);
    const float scale = __fdiv_rn(static_cast<float>(kBuckets), range);
    const bool bucketed = range > 0.f && scale <= 1e30f;
    int bsel = -1;              // bucket holding the threshold (-1: every candidate is in play)
    uint32_t k_left = topk;     // rank of the threshold among the keys in play
    uint32_t m = n_cand;        // keys in play
    if (bucketed) {
      // ---- 2. bucket histogram, then the bucket of the topk-th largest
      for (int g = 0; g < segments; ++g) {
#pragma unroll
        for (int c = 0; c < kRegChunks; ++c) {
          const float v = val_at(g, c);
          if (v != -INFINITY) atomicAdd(&hb[value_bucket(v, lo_half, scale)], 1u);
        }
      }
      __syncthreads();
      // thread i holds buckets 2047 - kBucketsPerThread i downwards; block scan in thread order
      uint32_t h4[kBucketsPerThread], s4 = 0;
#pragma unroll
      for (int e = 0; e < kBucketsPerThread; ++e) {
        h4[e] = hb[kBuckets - 1 - kBucketsPerThread * tid - e];
        s4 += h4[e];
      }
      uint32_t incl = s4;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) red_n[warp] = incl;
      __syncthreads();
      uint32_t before = 0;
      for (int w = 0; w < warp; ++w) before += red_n[w];
      incl += before;
      const uint32_t excl = incl - s4;
      if (incl >= topk && excl < topk) {
        uint32_t cum = excl, mb = 0;
        int eb = kBucketsPerThread - 1;
        bool found = false;
#pragma unroll
        for (int e = 0; e < kBucketsPerThread; ++e) {
          if (!found) {
            if (cum + h4[e] >= topk) {
              found = true;
              eb = e;
              mb = h4[e];
            } else {
              cum += h4[e];
            }
          }
        }
        bcast[0] = static_cast<uint32_t>(kBuckets - 1 - kBucketsPerThread * tid - eb);
        bcast[1] = cum;
        bcast[2] = mb;
      }
      __syncthreads();
      bsel = static_cast<int>(bcast[0]);
      k_left = topk - bcast[1];
      m = bcast[2];
    }
    if (bucketed && m <= static_cast<uint32_t>(kListCap)) {
      // ---- 3a. rank the keys of bucket bsel directly
      for (int g = 0; g < segments; ++g) {
#pragma unroll
        for (int c = 0; c < kRegChunks; ++c) {
          const float v = val_at(g, c);
          if (v != -INFINITY && value_bucket(v, lo_half, scale) == bsel) {
            const uint32_t slot = atomicAdd(&bcast[3], 1u);
            if (slot < static_cast<uint32_t>(kListCap)) list[slot] = score_key(v);
          }
        }
      }
      __syncthreads();
      if (static_cast<uint32_t>(tid) < m) {
        const uint32_t key = list[tid];
        uint32_t gt = 0, eq = 0;
        for (uint32_t i = 0; i < m; ++i) {
          const uint32_t o = list[i];
          gt += o > key ? 1u : 0u;
          eq += o == key ? 1u : 0u;
        }
        if (gt < k_left && k_left <= gt + eq) {  // every writer holds the same key
          bcast[4] = key;
          bcast[5] = k_left - gt;
        }
      }
      __syncthreads();
      T = bcast[4];
      k_rem = bcast[5];
    } else {
      // ---- 3b. byte-wise radix select over the keys in play
      uint32_t prefix = 0;
      for (int i = tid; i < 512; i += kSelThreads) hb[i] = 0;
      __syncthreads();
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        uint32_t* h = hb + (pass & 1) * 256;
        for (int g = 0; g < segments; ++g) {
#pragma unroll
          for (int c = 0; c < kRegChunks; ++c) {
            const float v = val_at(g, c);
            const uint32_t key = score_key(v);
            const bool in = key != 0u && (key & hi_mask) == prefix &&
                            (bsel < 0 || value_bucket(v, lo_half, scale) == bsel);
            if (__any_sync(0xffffffffu, in)) {
              const uint32_t bin = in ? ((key >> shift) & 0xFFu) : 256u;
              const uint32_t peers = __match_any_sync(0xffffffffu, bin);
              if (in && lane == __ffs(peers) - 1) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
            }
          }
        }
        __syncthreads();
        if (warp == 0) {
          // lane l sums bins 255-8l .. 248-8l (descending), then a scan across lanes
          uint32_t s8 = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) s8 += h[255 - 8 * lane - e];
          uint32_t inc = s8;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
          }
          const uint32_t exc = inc - s8;
          const uint32_t hit = __ballot_sync(0xffffffffu, inc >= k_left && exc < k_left);
          if (lane == __ffs(hit) - 1) {
            uint32_t cum = exc;
            int bin = 255 - 8 * lane;
            for (int e = 0; e < 8; ++e, --bin) {
              if (cum + h[bin] >= k_left) break;
              cum += h[bin];
            }
            bcast[6] = static_cast<uint32_t>(bin);
            bcast[7] = cum;
          }
        }
        // the other histogram is free: clear it for the next pass
        if (tid >= 256 && tid < 512) hb[((pass + 1) & 1) * 256 + tid - 256] = 0;
        __syncthreads();
        prefix |= bcast[6] << shift;
        k_left -= bcast[7];
      }
      T = prefix;
      k_rem = k_left;
    }
  }

  // ---- 4. compaction in position order, one segment of 8192 positions at a time
  uint32_t sel_run = 0, eq_run = 0;
  for (int g = 0; g < segments; ++g) {
#pragma unroll
    for (int c = 0; c < kRegChunks; ++c) {
      const uint32_t key = score_key(val_at(g, c));
      const uint32_t bg = __ballot_sync(0xffffffffu, key > T);
      const uint32_t be = __ballot_sync(0xffffffffu, key == T);
      if (lane == 0) {
        cnt[0][c * kSelWarps + warp] = __popc(bg);
        cnt[1][c * kSelWarps + warp] = __popc(be);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // 256 (chunk, warp) entries in position order, 8 consecutive ones per lane
      uint32_t gt[8], eq[8], s_eq = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        gt[e] = cnt[0][8 * lane + e];
        eq[e] = cnt[1][8 * lane + e];
        s_eq += eq[e];
      }
      uint32_t incl = s_eq;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      uint32_t eq_before = eq_run + incl - s_eq, s_sel = 0;
      uint32_t sel[8], eqb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t keep_eq = k_rem > eq_before ? min(k_rem - eq_before, eq[e]) : 0u;
        sel[e] = gt[e] + keep_eq;
        eqb[e] = eq_before;
        eq_before += eq[e];
        s_sel += sel[e];
      }
      uint32_t incl2 = s_sel;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += v;
      }
      uint32_t sel_before = sel_run + incl2 - s_sel;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[0][8 * lane + e] = sel_before;
        cnt[1][8 * lane + e] = eqb[e];
        sel_before += sel[e];
      }
      if (lane == 31) {
        bcast[2] = incl2;  // selected in this segment
        bcast[3] = incl;   // equal keys in this segment
      }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < kRegChunks; ++c) {
      const uint32_t key = score_key(val_at(g, c));
      const bool eqk = key == T;
      const uint32_t be = __ballot_sync(0xffffffffu, eqk);
      const uint32_t rank = cnt[1][c * kSelWarps + warp] + __popc(be & lt_mask);
      const bool sel = key > T || (eqk && rank < k_rem);
      const uint32_t bs = __ballot_sync(0xffffffffu, sel);
      const uint32_t pos = cnt[0][c * kSelWarps + warp] + __popc(bs & lt_mask);
      if (sel && pos < topk) out[pos] = g * kSelGroup + c * kSelThreads + tid;
    }
    sel_run += bcast[2];
    eq_run += bcast[3];
    __syncthreads();  // cnt and bcast are rewritten by the next segment
  }
  for (int i = static_cast<int>(min(sel_run, topk)) + tid; i < p.topk; i += kSelThreads) out[i] = -1;
}

}  // namespace mlaidx

// Scratch of mla_indexer_topk_noalloc: the fp32 scores of one call, in the
// library's own device image (the CUDA runtime creates it with the module), so
// that the call itself allocates nothing.  Its size is the call's limit:
// B * S1 * max_blocks_per_seq * 128 scores at most.  One array per device and
// process: calls that overlap in time (other streams, other host threads)
// share it and race.
constexpr size_t kNoAllocScratchFloats = size_t{2} << 20;  // 2 Mi fp32 = 8 MiB
static __device__ __align__(256) float g_idx_noalloc_scratch[kNoAllocScratchFloats];

// ==================================================================== C ABI
namespace {

thread_local char g_idx_error[512] = "";

mla_status idx_fail(mla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mla_status idx_fail(mla_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_idx_error, sizeof g_idx_error, fmt, ap);
  va_end(ap);
  return s;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

constexpr int kMaxDevices = 64;
std::once_flag g_attr_once[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
float* g_scratch_ptr[kMaxDevices];
cudaError_t g_attr_err[kMaxDevices];
int g_sm_count[kMaxDevices];

cudaError_t prepare(int dev) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
      g_encode_err = cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode_err != cudaSuccess) return g_encode_err;
  std::call_once(g_attr_once[dev], [dev] {
    cudaError_t e = cudaFuncSetAttribute(mlaidx::idx_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         mlaidx::kSmemMax);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    g_attr_err[dev] = e;
  });
  return g_attr_err[dev];
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

mla_status check_dims(const mla_indexer_dims* dims) {
  if (dims == nullptr) return idx_fail(MLA_ERR_NULL, "dims is NULL");
  const mla_indexer_dims d = *dims;
  if (d.B < 1 || d.S1 < 1 || d.topk < 1 || d.num_blocks < 1 || d.max_blocks_per_seq < 1)
    return idx_fail(MLA_ERR_SHAPE, "B, S1, topk, num_blocks and max_blocks_per_seq must be >= 1");
  if (d.B > 65535 || static_cast<int64_t>(d.B) * d.S1 > (1ll << 30))
    return idx_fail(MLA_ERR_SHAPE, "B=%d S1=%d too large", d.B, d.S1);
  if (d.head_dim != 128 || d.block_size != 128)
    return idx_fail(MLA_ERR_UNSUPPORTED, "head_dim=%d block_size=%d: only 128/128 are implemented", d.head_dim,
                    d.block_size);
  if (d.n_heads < 16 || d.n_heads % 16 != 0 || static_cast<int64_t>(d.S1) * d.n_heads > mlaidx::kMaxN)
    return idx_fail(MLA_ERR_UNSUPPORTED, "n_heads=%d S1=%d: n_heads must be a multiple of 16 and S1*n_heads <= %d",
                    d.n_heads, d.S1, mlaidx::kMaxN);
  if (static_cast<int64_t>(d.num_blocks) * 128 >= (1ll << 31))
    return idx_fail(MLA_ERR_SHAPE, "num_blocks=%d too large", d.num_blocks);
  if (static_cast<int64_t>(d.max_blocks_per_seq) * 128 >= (1ll << 31))
    return idx_fail(MLA_ERR_SHAPE, "max_blocks_per_seq=%d too large", d.max_blocks_per_seq);
  return MLA_OK;
}

size_t workspace_bytes(const mla_indexer_dims& d) {
  return static_cast<size_t>(d.B) * d.S1 * d.max_blocks_per_seq * 128 * sizeof(float);
}

// Checks shared by the score entry points; sets *dev and runs the per-device set-up.
mla_status check_score_args(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                            const int32_t* block_table, const int32_t* act_seqs, const void* scores,
                            size_t scores_bytes, int* dev) {
  const mla_status ds = check_dims(dims);
  if (ds != MLA_OK) return ds;
  const mla_indexer_dims d = *dims;
  if (!q || !w || !k_cache || !block_table || !act_seqs || !scores)
    return idx_fail(MLA_ERR_NULL, "a required pointer is NULL");
  if (scores_bytes < workspace_bytes(d))
    return idx_fail(MLA_ERR_SHAPE, "score buffer of %zu bytes, %zu needed", scores_bytes, workspace_bytes(d));
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(scores, 256) || !aligned(w, 4) ||
      !aligned(block_table, 4) || !aligned(act_seqs, 4))
    return idx_fail(MLA_ERR_ALIGN, "q/k_cache must be 16-byte, the score buffer 256-byte, the rest 4-byte aligned");
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return idx_fail(MLA_ERR_UNSUPPORTED, "device ordinal %d too large", *dev);
  e = prepare(*dev);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "set-up: %s", cudaGetErrorString(e));
  return MLA_OK;
}

mla_status check_select_args(const mla_indexer_dims* dims, const float* scores, const int32_t* act_seqs,
                             const int32_t* topk_idx) {
  const mla_status ds = check_dims(dims);
  if (ds != MLA_OK) return ds;
  if (!scores || !act_seqs || !topk_idx) return idx_fail(MLA_ERR_NULL, "a required pointer is NULL");
  if (!aligned(scores, 4) || !aligned(act_seqs, 4) || !aligned(topk_idx, 4))
    return idx_fail(MLA_ERR_ALIGN, "scores, act_seqs and topk_idx must be 4-byte aligned");
  return MLA_OK;
}

// Launches the score kernel (arguments already checked).
mla_status launch_scores(const mla_indexer_dims& d, int dev, const void* q, const float* w, const void* k_cache,
                         const int32_t* block_table, const int32_t* act_seqs, float* scores, cudaStream_t s) {
  // tensor map over the key cache: rows x 128 dims of bf16, boxes of 128 rows x 64 dims, 128-byte swizzle
  CUtensorMap kmap;
  const cuuint64_t gdim[2] = {128, static_cast<cuuint64_t>(d.num_blocks) * 128};
  const cuuint64_t gstride[1] = {128 * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult cr = g_encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k_cache), gdim, gstride,
                               box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return idx_fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(cr));
  // tensor map over q: (token, head) rows x 128 dims; one box = one sequence's S1 * H rows x 64 dims
  CUtensorMap qmap;
  const cuuint64_t qdim[2] = {128, static_cast<cuuint64_t>(d.B) * d.S1 * d.n_heads};
  const cuuint32_t qbox[2] = {64, static_cast<cuuint32_t>(d.S1 * d.n_heads)};
  const CUresult qr = g_encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), qdim, gstride, qbox,
                               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (qr != CUDA_SUCCESS) return idx_fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", static_cast<int>(qr));

  mlaidx::ScoreParams sp;
  sp.q = static_cast<const uint16_t*>(q);
  sp.w = w;
  sp.block_table = block_table;
  sp.act_seqs = act_seqs;
  sp.scores = scores;
  sp.ld = static_cast<int64_t>(d.max_blocks_per_seq) * 128;
  sp.S1 = d.S1;
  sp.H = d.n_heads;
  sp.N = d.S1 * d.n_heads;
  sp.num_blocks = d.num_blocks;
  sp.mbps = d.max_blocks_per_seq;
  // as many N-column accumulators as fit in the 512 TMEM columns, up to kMaxAcc
  sp.n_acc = 512 / sp.N < mlaidx::kMaxAcc ? 512 / sp.N : mlaidx::kMaxAcc;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(sp.n_acc * sp.N)) cols <<= 1;
  sp.tmem_cols = cols;
  sp.wait_ns = mlasp::host_wait_limit_ns();
  // about one wave: split each sequence's tiles over SMs / B CTAs
  const int per_b = g_sm_count[dev] / d.B > 1 ? g_sm_count[dev] / d.B : 1;
  sp.tiles_per_cta = (d.max_blocks_per_seq + per_b - 1) / per_b;
  const dim3 grid(static_cast<unsigned>((d.max_blocks_per_seq + sp.tiles_per_cta - 1) / sp.tiles_per_cta),
                  static_cast<unsigned>(d.B));
  // Q chunks of N rows, then as many 32 KB key stages as fit
  sp.q_chunk = static_cast<uint32_t>(sp.N) * 128;
  sp.off_stages = (mlaidx::kOffQ + 2 * sp.q_chunk + 1023u) & ~1023u;
  sp.stages = static_cast<int>((mlaidx::kSmemMax - sp.off_stages) / mlaidx::kTileBytes);
  if (sp.stages > mlaidx::kMaxStages) sp.stages = mlaidx::kMaxStages;
  const size_t smem_bytes = sp.off_stages + static_cast<size_t>(sp.stages) * mlaidx::kTileBytes;
  mlaidx::idx_scores_kernel<<<grid, mlaidx::kThreads, smem_bytes, s>>>(kmap, qmap, sp);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "score kernel launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}

// Launches the selection kernel (arguments already checked).  `behind_scores`:
// it directly follows the score kernel on `s`, so it may be launched as a
// programmatic dependent (its launch overlaps the score grid's tail).
mla_status launch_select(const mla_indexer_dims& d, const float* scores, const int32_t* act_seqs, int32_t* topk_idx,
                         cudaStream_t s, bool behind_scores) {
  mlaidx::SelectParams sel;
  sel.scores = scores;
  sel.ld = static_cast<int64_t>(d.max_blocks_per_seq) * 128;
  sel.S1 = d.S1;
  sel.act_seqs = act_seqs;
  sel.topk_idx = topk_idx;
  sel.topk = d.topk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(d.B * d.S1), 1, 1);
  cfg.blockDim = dim3(mlaidx::kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = behind_scores ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, mlaidx::idx_topk_kernel, sel);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "selection kernel launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_indexer_workspace_bytes(const mla_indexer_dims* dims) {
  if (check_dims(dims) != MLA_OK) return 0;
  return workspace_bytes(*dims);
}

mla_status mla_indexer_scores(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                              const int32_t* block_table, const int32_t* act_seqs, float* scores,
                              size_t scores_bytes, void* stream) {
  g_idx_error[0] = '\0';
  int dev = 0;
  const mla_status st = check_score_args(dims, q, w, k_cache, block_table, act_seqs, scores, scores_bytes, &dev);
  if (st != MLA_OK) return st;
  return launch_scores(*dims, dev, q, w, k_cache, block_table, act_seqs, scores, static_cast<cudaStream_t>(stream));
}

mla_status mla_indexer_select(const mla_indexer_dims* dims, const float* scores, const int32_t* act_seqs,
                              int32_t* topk_idx, void* stream) {
  g_idx_error[0] = '\0';
  const mla_status st = check_select_args(dims, scores, act_seqs, topk_idx);
  if (st != MLA_OK) return st;
  return launch_select(*dims, scores, act_seqs, topk_idx, static_cast<cudaStream_t>(stream), false);
}

mla_status mla_indexer_topk(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                            const int32_t* block_table, const int32_t* act_seqs, int32_t* topk_idx,
                            void* workspace, size_t ws_bytes, void* stream) {
  g_idx_error[0] = '\0';
  int dev = 0;
  mla_status st = check_score_args(dims, q, w, k_cache, block_table, act_seqs, workspace, ws_bytes, &dev);
  if (st == MLA_OK) st = check_select_args(dims, static_cast<const float*>(workspace), act_seqs, topk_idx);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* scores = static_cast<float*>(workspace);
  st = launch_scores(*dims, dev, q, w, k_cache, block_table, act_seqs, scores, s);
  if (st != MLA_OK) return st;
  return launch_select(*dims, scores, act_seqs, topk_idx, s, true);
}

// For callers that cannot allocate device memory at call time, e.g. a host
// program that sizes all its device memory once at start-up, where a later
// cudaMalloc could fail or wait for the whole device.  Same work as
// mla_indexer_topk; the scores go to g_idx_noalloc_scratch instead of a
// caller workspace.  The first call on a device looks the array's address up
// (cudaGetSymbolAddress) and keeps it; nothing else is set up.
mla_status mla_indexer_topk_noalloc(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                                    const int32_t* block_table, const int32_t* act_seqs, int32_t* topk_idx,
                                    void* stream) {
  g_idx_error[0] = '\0';
  const mla_status ds = check_dims(dims);
  if (ds != MLA_OK) return ds;
  const size_t need = workspace_bytes(*dims);
  if (need > sizeof(float) * kNoAllocScratchFloats)
    return idx_fail(MLA_ERR_SHAPE,
                    "B * S1 * max_blocks_per_seq * 128 = %zu scores exceed the no-allocation scratch of %zu scores; "
                    "use mla_indexer_topk with a workspace",
                    need / sizeof(float), kNoAllocScratchFloats);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return idx_fail(MLA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  std::call_once(g_scratch_once[dev], [dev] {
    void* ptr = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&ptr, g_idx_noalloc_scratch);
    g_scratch_ptr[dev] = static_cast<float*>(ptr);
  });
  if (g_scratch_err[dev] != cudaSuccess)
    return idx_fail(MLA_ERR_CUDA, "cudaGetSymbolAddress of the scratch: %s", cudaGetErrorString(g_scratch_err[dev]));
  float* scratch = g_scratch_ptr[dev];
  // Nothing in the scratch has to start at zero: the score phase writes every
  // position below act_seqs[b] before the selection phase of the same call
  // reads it, and neither reads beyond.
  int dev2 = 0;
  mla_status st = check_score_args(dims, q, w, k_cache, block_table, act_seqs, scratch, need, &dev2);
  if (st == MLA_OK) st = check_select_args(dims, scratch, act_seqs, topk_idx);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_scores(*dims, dev2, q, w, k_cache, block_table, act_seqs, scratch, s);
  if (st != MLA_OK) return st;
  return launch_select(*dims, scratch, act_seqs, topk_idx, s, true);
}

mla_status mla_indexer_device_status(void* stream, uint32_t* flags, int32_t clear) {
  g_idx_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, mlaidx::g_idx_status, sizeof v);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(mlaidx::g_idx_status, &zero, sizeof zero);
    if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  if (flags) *flags = v;
  if (v != 0) return idx_fail(MLA_ERR_DEVICE_STATUS, "indexer device status 0x%x", v);
  return MLA_OK;
}

const char* mla_indexer_last_error(void) { return g_idx_error; }

}  // extern "C"
