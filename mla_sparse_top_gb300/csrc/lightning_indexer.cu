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
// weighted ReLU sum over heads is thread-local.  TMEM holds two accumulators,
// so the epilogue of tile i overlaps the MMA of tile i + 1.
//   warp 0      TMA producer (one thread), 4-stage key ring
//   warp 1      TMEM allocation and MMA issue (one thread)
//   warps 2-3   load the sequence's Q rows and head weights once
//   warps 4-7   epilogue: ReLU, weights, head sum, fp32 scores to the workspace
//
// Kernel 2 (selection), one CTA per token: an exact radix select on the
// order-preserving 32-bit image of the fp32 scores (four 8-bit passes) finds
// the k-th largest key T and how many entries equal to T are kept; a
// compaction in position order then writes the positions with key > T and the
// first ones with key == T, so the output is ascending and ties go to the
// smaller position.
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

namespace mlaidx {
using namespace mlasp;

constexpr int kBlock = 128;                  // keys per tile = rows per cache block
constexpr int kDim = 128;                    // head_dim
constexpr int kStages = 4;
constexpr int kChunkBytes = kBlock * 128;    // 128 rows x 64 bf16 dims (128-byte swizzled rows)
constexpr int kTileBytes = 2 * kChunkBytes;  // 32 KB
constexpr int kMaxN = 256;                   // S1 * H
constexpr int kQChunkBytes = kMaxN * 128;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 128;

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kTileBytes;
constexpr int kOffW = kOffQ + 2 * kQChunkBytes;
constexpr int kOffBars = kOffW + kMaxN * 4;
constexpr int kBarFull = 0;                  // [kStages]
constexpr int kBarEmpty = kBarFull + kStages;  // [kStages]
constexpr int kBarTFull = kBarEmpty + kStages;  // [2]
constexpr int kBarTEmpty = kBarTFull + 2;    // [2]
constexpr int kBarQReady = kBarTEmpty + 2;
constexpr int kBarFinal = kBarQReady + 1;    // the MMA thread's last commit
constexpr int kNumBars = kBarFinal + 1;
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kSmemBytes = kOffAbort + 4;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kQChunkBytes % 1024 == 0 && kTileBytes % 1024 == 0, "operand alignment");

constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

__device__ unsigned int g_idx_status = 0;

struct ScoreParams {
  const uint16_t* q;
  const float* w;
  const int32_t* block_table;
  const int32_t* act_seqs;
  float* scores;
  int64_t ld;  // scores row stride (floats)
  int S1, H, N, num_blocks, mbps, tiles_per_cta;
  uint32_t tmem_cols;
};

struct Ctx {
  uint32_t sbase;
  uint8_t* smem;
  volatile uint32_t* abort;
  __device__ uint32_t bar(int i) const { return sbase + kOffBars + 8 * i; }
};

__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity) {
  return mbar_wait<false>(c.bar(idx), parity, c.abort, kWaitLimitNs);
}
__device__ __forceinline__ bool warp_wait(const Ctx& c, int idx, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(c, idx, parity));
}

// 2-D TMA tiled load (box of the tensor map at coordinates {x, y}) into
// shared memory, counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
idx_scores_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ ScoreParams p) {
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
  if (tid == 0) {
    const bool misaligned = (c.sbase & 1023u) != 0;
    *c.abort = ((*reinterpret_cast<volatile unsigned int*>(&g_idx_status) & MLA_DEVICE_TIMEOUT) || misaligned) ? 1u : 0u;
    if (misaligned) atomicOr(&g_idx_status, MLA_DEVICE_TIMEOUT);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(c.bar(kBarFull + i), 1);
      mbar_init(c.bar(kBarEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(c.bar(kBarTFull + i), 1);
      mbar_init(c.bar(kBarTEmpty + i), kEpiThreads);
    }
    mbar_init(c.bar(kBarQReady), 64);
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
  const int64_t qrow0 = static_cast<int64_t>(b) * p.N;  // the sequence's (token, head) rows are contiguous

  if (!*c.abort) {
    if (warp == 0) {
      // ---- TMA producer
      if (lane == 0) {
        for (int i = 0; i < ntile; ++i) {
          const int st = i % kStages;
          if (!wait_bar(c, kBarEmpty + st, ((i / kStages) & 1) ^ 1)) break;
          const int blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.mbps + tile0 + i);
          if (blk >= 0 && blk < p.num_blocks) {
            const uint32_t dst = c.sbase + kOffStages + st * kTileBytes;
            mbar_arrive_expect_tx(c.bar(kBarFull + st), kTileBytes);
            tma_load_2d(dst, &kmap, 0, blk * kBlock, c.bar(kBarFull + st));
            tma_load_2d(dst + kChunkBytes, &kmap, 64, blk * kBlock, c.bar(kBarFull + st));
          } else {
            // not a candidate block: the epilogue writes -inf for its keys
            atomicOr(&g_idx_status, MLA_DEVICE_BAD_BLOCK);
            mbar_arrive(c.bar(kBarFull + st));
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---- MMA issue
      if (lane == 0 && wait_bar(c, kBarQReady, 0)) {
        const uint32_t idesc = make_idesc_f16(128, static_cast<uint32_t>(p.N), 1, 0, 0);
        for (int i = 0; i < ntile; ++i) {
          const int st = i % kStages, buf = i & 1;
          if (!wait_bar(c, kBarFull + st, (i / kStages) & 1)) break;
          if (!wait_bar(c, kBarTEmpty + buf, ((i >> 1) & 1) ^ 1)) break;
          tc_fence_after();
          const uint32_t a0 = c.sbase + kOffStages + st * kTileBytes;
          const uint32_t b0 = c.sbase + kOffQ;
          const uint32_t d = tmem + static_cast<uint32_t>(buf * p.N);
#pragma unroll
          for (int s = 0; s < 8; ++s)
            umma_ss(d, make_sdesc(a0 + (s >> 2) * kChunkBytes + (s & 3) * 32, 16, 1024, kSwizzle128B),
                    make_sdesc(b0 + (s >> 2) * kQChunkBytes + (s & 3) * 32, 16, 1024, kSwizzle128B), idesc,
                    s > 0 ? 1u : 0u);
          umma_commit(c.bar(kBarTFull + buf));
          umma_commit(c.bar(kBarEmpty + st));
        }
      }
      if (lane == 0) {
        // no MMA may still run when TMEM is released, even after an abort
        umma_commit(c.bar(kBarFinal));
        volatile uint32_t never = 0;
        mbar_wait<false>(c.bar(kBarFinal), 0, &never, kWaitLimitNs);
      }
      __syncwarp();
    } else if (warp < kEpiWarp0) {
      // ---- Q rows (N x 128 dims, bf16) and head weights, once
      const int t2 = tid - 64;
      const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(p.q) + qrow0 * kDim * 2;
      for (int ui = t2; ui < p.N * 16; ui += 64) {
        const int n = ui >> 4, du = ui & 15, ch = du >> 3, u = du & 7;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(qsrc + static_cast<int64_t>(n) * kDim * 2 + du * 16));
        const uint32_t dst = c.sbase + kOffQ + ch * kQChunkBytes + n * 128 + ((u ^ (n & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      float* wsm = reinterpret_cast<float*>(smem + kOffW);
      for (int n = t2; n < p.N; n += 64) wsm[n] = __ldg(p.w + qrow0 + n);
      fence_proxy_async_smem();
      mbar_arrive(c.bar(kBarQReady));
    } else {
      // ---- epilogue: thread = key (TMEM lane)
      const int q4 = warp - kEpiWarp0;
      const int kin = q4 * 32 + lane;
      const float* wsm = reinterpret_cast<const float*>(smem + kOffW);
      const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
      const bool have_w = warp_wait(c, kBarQReady, 0);  // the weights are in shared memory
      for (int i = 0; have_w && i < ntile; ++i) {
        const int buf = i & 1, tl = tile0 + i;
        if (!warp_wait(c, kBarTFull + buf, (i >> 1) & 1)) break;
        tc_fence_after();
        const int blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.mbps + tl);
        const bool valid_blk = blk >= 0 && blk < p.num_blocks;
        const int j = tl * kBlock + kin;
        const uint32_t d = tmem + lane_off + static_cast<uint32_t>(buf * p.N);
        for (int s = 0; s < p.S1; ++s) {
          float acc = 0.f;
          for (int h0 = 0; h0 < p.H; h0 += 16) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(d + static_cast<uint32_t>(s * p.H + h0), v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) acc = fmaf(wsm[s * p.H + h0 + e], fmaxf(__uint_as_float(v[e]), 0.f), acc);
          }
          if (j < act) p.scores[(static_cast<int64_t>(b) * p.S1 + s) * p.ld + j] = valid_blk ? acc : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(c.bar(kBarTEmpty + buf));
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
constexpr int kSelThreads = 512;

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
// every finite score; it is treated as key 0 instead.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = f == 0.f ? 0u : __float_as_uint(f);
  if (f == -INFINITY) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads) idx_topk_kernel(const SelectParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sum[kSelThreads / 32][2];
  __shared__ uint32_t bcast[4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int act = __ldg(p.act_seqs + t / p.S1);
  // positions past the block table's width have no block: not candidates
  if (tid == 0 && static_cast<int64_t>(act) > p.ld) atomicOr(&g_idx_status, MLA_DEVICE_BAD_BLOCK);
  const int n = static_cast<int>(min(static_cast<int64_t>(max(act, 0)), p.ld));
  const float* row = p.scores + static_cast<int64_t>(t) * p.ld;
  int32_t* out = p.topk_idx + static_cast<int64_t>(t) * p.topk;

  // candidates (key != 0)
  uint32_t cnt = 0;
  for (int j = tid; j < n; j += kSelThreads) cnt += score_key(__ldg(row + j)) != 0u;
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) warp_sum[warp][0] = cnt;
  __syncthreads();
  if (tid == 0) {
    uint32_t tot = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) tot += warp_sum[w][0];
    bcast[0] = tot;
  }
  __syncthreads();
  const uint32_t n_cand = bcast[0];

  // threshold key T and how many entries equal to T are kept
  uint32_t T = 0, k_rem = 0;
  if (n_cand > static_cast<uint32_t>(p.topk)) {
    uint32_t prefix = 0;
    k_rem = static_cast<uint32_t>(p.topk);
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      const uint32_t hi_mask = shift == 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
      for (int j = tid; j < n; j += kSelThreads) {
        const uint32_t k = score_key(__ldg(row + j));
        if ((k & hi_mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l sums bins 255-8l .. 248-8l (descending), then a scan across lanes
        uint32_t s8 = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) s8 += hist[255 - 8 * lane - e];
        uint32_t incl = s8;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - s8;
        const uint32_t hit = __ballot_sync(0xffffffffu, incl >= k_rem && excl < k_rem);
        const int src = __ffs(hit) - 1;
        if (lane == src) {
          uint32_t cum = excl;
          int bin = 255 - 8 * lane;
          for (int e = 0; e < 8; ++e, --bin) {
            if (cum + hist[bin] >= k_rem) break;
            cum += hist[bin];
          }
          bcast[1] = static_cast<uint32_t>(bin);
          bcast[2] = cum;
        }
      }
      __syncthreads();
      prefix |= bcast[1] << shift;
      k_rem -= bcast[2];
      __syncthreads();
    }
    T = prefix;
  }

  // compaction in position order: key > T, or key == T among the first k_rem
  uint32_t sel_base = 0, eq_base = 0;
  for (int j0 = 0; j0 < n; j0 += kSelThreads) {
    const int j = j0 + tid;
    const uint32_t k = j < n ? score_key(__ldg(row + j)) : 0u;
    const bool eq = j < n && k == T && k != 0u;
    const uint32_t eq_bits = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_sum[warp][0] = __popc(eq_bits);
    __syncthreads();
    uint32_t eq_before = eq_base, eq_tot = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) {
      if (w < warp) eq_before += warp_sum[w][0];
      eq_tot += warp_sum[w][0];
    }
    eq_before += __popc(eq_bits & ((1u << lane) - 1u));
    const bool sel = j < n && k != 0u && (k > T || (eq && eq_before < k_rem));
    const uint32_t sel_bits = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) warp_sum[warp][1] = __popc(sel_bits);
    __syncthreads();
    uint32_t sel_before = sel_base, sel_tot = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) {
      if (w < warp) sel_before += warp_sum[w][1];
      sel_tot += warp_sum[w][1];
    }
    sel_before += __popc(sel_bits & ((1u << lane) - 1u));
    if (sel && sel_before < static_cast<uint32_t>(p.topk)) out[sel_before] = j;
    sel_base += sel_tot;
    eq_base += eq_tot;
    __syncthreads();
  }
  for (int i = static_cast<int>(min(sel_base, static_cast<uint32_t>(p.topk))) + tid; i < p.topk; i += kSelThreads)
    out[i] = -1;
}

}  // namespace mlaidx

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
                                         mlaidx::kSmemBytes);
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

}  // namespace

extern "C" {

size_t mla_indexer_workspace_bytes(const mla_indexer_dims* dims) {
  if (check_dims(dims) != MLA_OK) return 0;
  return workspace_bytes(*dims);
}

mla_status mla_indexer_topk(const mla_indexer_dims* dims, const void* q, const float* w, const void* k_cache,
                            const int32_t* block_table, const int32_t* act_seqs, int32_t* topk_idx,
                            void* workspace, size_t ws_bytes, void* stream) {
  g_idx_error[0] = '\0';
  const mla_status ds = check_dims(dims);
  if (ds != MLA_OK) return ds;
  const mla_indexer_dims d = *dims;
  if (!q || !w || !k_cache || !block_table || !act_seqs || !topk_idx || !workspace)
    return idx_fail(MLA_ERR_NULL, "a required pointer is NULL");
  if (ws_bytes < workspace_bytes(d))
    return idx_fail(MLA_ERR_SHAPE, "workspace of %zu bytes, %zu needed", ws_bytes, workspace_bytes(d));
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(workspace, 256) || !aligned(w, 4) ||
      !aligned(block_table, 4) || !aligned(act_seqs, 4) || !aligned(topk_idx, 4))
    return idx_fail(MLA_ERR_ALIGN, "q/k_cache must be 16-byte, workspace 256-byte, the rest 4-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return idx_fail(MLA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  e = prepare(dev);
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "set-up: %s", cudaGetErrorString(e));

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

  mlaidx::ScoreParams sp;
  sp.q = static_cast<const uint16_t*>(q);
  sp.w = w;
  sp.block_table = block_table;
  sp.act_seqs = act_seqs;
  sp.scores = static_cast<float*>(workspace);
  sp.ld = static_cast<int64_t>(d.max_blocks_per_seq) * 128;
  sp.S1 = d.S1;
  sp.H = d.n_heads;
  sp.N = d.S1 * d.n_heads;
  sp.num_blocks = d.num_blocks;
  sp.mbps = d.max_blocks_per_seq;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * sp.N)) cols <<= 1;
  sp.tmem_cols = cols;
  // about one wave: split each sequence's tiles over SMs / B CTAs
  const int per_b = g_sm_count[dev] / d.B > 1 ? g_sm_count[dev] / d.B : 1;
  sp.tiles_per_cta = (d.max_blocks_per_seq + per_b - 1) / per_b;
  const dim3 grid1(static_cast<unsigned>((d.max_blocks_per_seq + sp.tiles_per_cta - 1) / sp.tiles_per_cta),
                   static_cast<unsigned>(d.B));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mlaidx::idx_scores_kernel<<<grid1, mlaidx::kThreads, mlaidx::kSmemBytes, s>>>(kmap, sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "score kernel launch: %s", cudaGetErrorString(e));

  mlaidx::SelectParams sel;
  sel.scores = static_cast<const float*>(workspace);
  sel.ld = sp.ld;
  sel.S1 = d.S1;
  sel.act_seqs = act_seqs;
  sel.topk_idx = topk_idx;
  sel.topk = d.topk;
  mlaidx::idx_topk_kernel<<<static_cast<unsigned>(d.B * d.S1), mlaidx::kSelThreads, 0, s>>>(sel);
  e = cudaGetLastError();
  if (e != cudaSuccess) return idx_fail(MLA_ERR_CUDA, "selection kernel launch: %s", cudaGetErrorString(e));
  return MLA_OK;
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
