// Fused sparse MLA attention forward for GB300 (sm_103a).
//
// One query token is processed by a cluster of two CTAs.  CTA r (its rank in
// the cluster) owns the latent dims [256r, 256r+256) and the rope dims
// [32r, 32r+32): it gathers only that half of every selected cache row, so
// every byte is read once, and it accumulates O[:, its 256 latent dims] for
// all 128 heads in tensor memory (O for a whole token is 128 x 512 fp32 =
// 256 KB, the entire TMEM of one SM, which is why a token needs two SMs).
// Scores need all 576 dims: each CTA computes a partial score tile over its
// 288 dims and sends it (fp32) to the peer through distributed shared memory;
// both CTAs then hold bit-identical score tiles (fp32 addition commutes) and
// run the same online softmax.  Dedicated warps stage the partial tile in
// local shared memory and hand it to the TMA engine as bulk copies into the
// peer, so the CTA-to-CTA traffic never queues in front of other warps'
// shared-memory accesses.  Each side reads its partial score tile out of
// TMEM at once, so the next score MMA overlaps with the exchange.
//
// Per CTA (24 warps; registers rebalanced per warpgroup with setmaxnreg):
//   warps 0-7   softmax: TMEM lane h = head h; warps w and w+4 share the
//               lanes of quadrant w % 4 and take key columns [32c, 32c+32),
//               c = w / 4.  Per tile read the own partial S,
//               add the peer's, mask and scale, row max across the warp pair,
//               lazy online softmax, write P over S in its TMEM region as
//               P_hi = bf16(p), P_lo = bf16(p - P_hi); final O / l -> bf16, lse.
//   warps 8-11  senders: partial S tile -> staging buffer -> bulk copies to
//               the peer, one 32-key column half at a time; each token's Q
//               (latent dims [0, 128) into TMEM, [128, 256) and the rope dims
//               into smem) as soon as the previous token's score MMAs are
//               complete (INT8 instantiations: the softmax warps load Q).
//   warps 12-19 gather: all eight warps on every key tile (8 keys each); bf16
//               cache by cp.async with zero fill for masked entries, INT8
//               cache by loads, dequantisation to bf16 and stores.
//   warp 20     MMA issue (one thread, polling both hand-offs): S = Q K^T
//               (A = Q latent in TMEM, rope in smem) and O += P_hi V + P_lo V
//               (A = P in TMEM, B = V MN-major), each as soon as it is ready.
//   warps 21-22 index resolution: topk entry -> validity -> block_table -> row.
//
// The stages follow "DeepSeek V3/V2 Sparse Flash Attention with Quantization",
// section "Compute pipeline" (Sa_V0 gather + INT8 dequant, Sa_C1 S = Q K^T,
// Sa_V1 softmax(S * scale), Sa_C2 O = P V, Sa_V2 O = o / l on the last tile)
// with the running (m, l, o) update of its section "Flash online softmax
// incremental update".
//
// Precision: every product is exact (bf16 x bf16 into fp32).  P enters the
// P.V product as two bf16 terms, so its relative error stays below 2^-18 and
// the result meets the stated tolerance of the exact definition even when a
// few keys carry the weight (P rounded once to bf16 or fp16 does not).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/mla_sparse.h"
#include "ptx.cuh"

namespace mlasp {

// ------------------------------------------------------------------ layout
constexpr int kThreads = 768;
constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kSenderWarp0 = 8;
constexpr int kSenderThreads = 128;
constexpr int kGatherWarp0 = 12;
constexpr int kMmaWarp = 20;
constexpr int kIndexWarp = 21;   // warps 21 and 22
constexpr int kIndexWarps = 2;
constexpr int kIdxBatch = 4;     // tiles resolved per index-warp pass
// register shares (launch: 768 threads x 80 registers = 61,440)
template <bool kInt8>
struct Regs {
  static constexpr uint32_t kSoftmax = kInt8 ? 120 : 136;
  static constexpr uint32_t kGather = kInt8 ? 56 : 40;
  static constexpr uint32_t kControl = 48;
  static_assert(256 * kSoftmax + 128 * 80 + 256 * kGather + 128 * kControl <= 768 * 80, "register budget");
};

constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr int kRegions = 3;  // TMEM score/P regions: tiles i, i+1, i+2 in flight
constexpr int kIdxSlots = kIndexWarps * kIdxBatch;
constexpr int kHeads = 128;
constexpr int kChunkBytes = kTileKeys * 128;            // 64 keys x 64 bf16 latent dims (128-byte swizzle)
constexpr int kRopeChunkBytes = kTileKeys * 64;         // 64 keys x 32 bf16 rope dims (64-byte swizzle)
constexpr int kStageBytes = 4 * kChunkBytes + kRopeChunkBytes;
constexpr int kXchgBytes = kHeads * 32 * 4;            // one column half (32 keys) of an fp32 partial score tile
constexpr int kXchgBlockBytes = 32 * 32 * 4;           // its 32 heads of one TMEM lane quadrant: one bulk copy
constexpr int kQHalfBytes = kHeads * 128 * 2;          // Q latent dims [128, 256) of this CTA (bf16)
constexpr int kQRopeBytes = kHeads * 64;

constexpr int kOffRecv = 0;                            // [2] one slot per column half, same offset in both CTAs
constexpr int kOffStaging = kOffRecv + 2 * kXchgBytes;  // [2] one staging buffer per column half
constexpr int kOffStages = kOffStaging + 2 * kXchgBytes;
constexpr int kOffQHalf = kOffStages + kStages * kStageBytes;
constexpr int kOffQRope = kOffQHalf + kQHalfBytes;
constexpr int kOffRows = kOffQRope + kQRopeBytes;       // int32 [kIdxSlots][64]
constexpr int kOffPair = kOffRows + kIdxSlots * kTileKeys * 4;
constexpr int kOffVmask = kOffPair + 4 * kHeads * 4;    // uint64 [kStages]; the pair slots are float [2][2][kHeads]
constexpr int kOffBars = kOffVmask + kStages * 8;
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarIdxFull = kBarEmpty + kStages;
constexpr int kBarIdxEmpty = kBarIdxFull + kIdxSlots;
// tile i uses TMEM region i % kRegions and barrier [i % kRegions] of each set
constexpr int kBarSFull = kBarIdxEmpty + kIdxSlots;      // [kRegions] S(i) computed
constexpr int kBarSFree = kBarSFull + kRegions;          // [kRegions] senders have read S(i)
constexpr int kBarPFull = kBarSFree + kRegions;          // [kRegions] P(i) written
constexpr int kBarPvDone = kBarPFull + kRegions;         // [kRegions] P(i).V accumulated
// Each column half has its own receive slot: column half c of tile i lands
// in slot c as phase i of RecvFull[c]; once the four softmax warps of that
// half have read it, phase i of PeerFree[c] (in the sending CTA) completes, and
// half c of tile i + 1 may be sent.  The two halves of a tile travel
// independently.  Every waiter waits for phase i of a barrier whose phase
// i - 1 is already complete, so the parity test is unambiguous.
constexpr int kBarRecvFull = kBarPvDone + kRegions;      // [2]
constexpr int kBarPeerFree = kBarRecvFull + 2;           // [2]
constexpr int kBarPairA = kBarPeerFree + 2;              // [4]
constexpr int kBarQReady = kBarPairA + 4;   // phase m: Q of the cluster's m-th token is loaded
constexpr int kBarQFree = kBarQReady + 1;    // phase m: the score MMAs of the m-th token are complete
constexpr int kBarOFree = kBarQFree + 1;     // phase m: O of the m-th token has been read out
constexpr int kBarFinal = kBarOFree + 1;
constexpr int kNumBars = kBarFinal + 1;
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffZero = kOffAbort + 4;  // a zero the compiler cannot see (dependency anchor)
constexpr int kOffTotal = kOffZero + 4;  // the cluster's tile count (read where registers are short)
constexpr int kSmemBytes = kOffTotal + 4;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStages % 1024 == 0 && kStageBytes % 1024 == 0 && kOffQHalf % 1024 == 0 && kOffQRope % 512 == 0,
              "operand alignment");
static_assert(kOffStaging % 16 == 0 && kXchgBlockBytes % 16 == 0, "bulk copy alignment");
static_assert(kOffBars % 8 == 0, "barrier alignment");

// TMEM columns (512 allocated): O | regions 0..2 | Q latent dims [0, 128) of
// this CTA (bf16 pairs; dims [128, 256) are a shared-memory operand).  Tile
// i's score tile S(i) (64 fp32 columns) lands in region i % 3; once it has
// been read out, P(i) overwrites it as P_hi (columns 0-31 of the region) and
// P_lo (columns 32-63), each 64 bf16 keys per row.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemRegion = 256;  // + 64 * (i % kRegions)
constexpr uint32_t kTmemQ = 448;
static_assert(kTmemRegion + 64 * kRegions <= kTmemQ && kTmemQ + 64 == kTmemCols, "TMEM layout");

// Partial result of a cut token (one CTA rank's 256 latent dims): O as float4
// units [(half * 32 + u) * 128 + h] (head h, dims 128 half + 4u .. + 3, so a
// warp's 32 heads store 512 contiguous bytes), then m[128] and l[128].
constexpr int kSlotFloats = kHeads * 256 + 2 * kHeads;

__device__ unsigned int g_mla_status = 0;

struct Params {
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  const void* kv_nope;
  const uint16_t* kv_rope;
  const float* kv_scales;
  const int32_t* topk_idx;
  const int32_t* block_table;
  const int32_t* act_seqs;
  uint16_t* out;
  float* lse;
  int S1, n_q, topk, num_blocks, mbps, n_tiles;
  int T;           // query tokens B * S1
  // Persistent clusters walk a stream of (token, tile) pairs.  Whole tokens:
  // cluster c takes tokens c, c + n_clusters, ... (the tokens of one sequence
  // run side by side on neighbouring clusters, so rows their lists share are
  // read from HBM once).  Equal shares (list mode kModeListsCut): cluster c
  // takes the tiles [c U / n_clusters, (c + 1) U / n_clusters) of
  // g = t * n_tiles + i, U = T * n_tiles; a token cut between clusters leaves
  // one partial softmax state per part in `ws`, merged by combine_kernel.
  int n_clusters;
  float* ws;  // equal shares: [n_clusters][2 segments][2 ranks] partial states (kSlotFloats each)
  int window;      // > 0: sliding window of this many positions instead of top-k lists
  // compressed cache (mode 2): entries after the window are compressed entries
  const void* cmp_nope;
  const uint16_t* cmp_rope;
  const float* cmp_scales;
  const int32_t* cmp_block_table;
  const int32_t* cmp_idx;  // SCFA lists [T, cmp_topk]; nullptr: CFA (every visible entry)
  int cmp_num_blocks, cmp_mbps, cmp_ratio, cmp_topk;
  float scale_log2;
  unsigned long long wait_ns;  // bound of every wait
  int out32;  // out is 32-byte aligned: the epilogue stores 32 bytes per instruction
};

struct Ctx {
  uint32_t sbase;
  uint8_t* smem;
  uint32_t tmem;
  uint32_t crank;
  int cid;        // cluster index
  int first;      // equal shares: tile g = t * n_tiles + i at the cluster's position 0 (T * n_tiles < 2^31)
  int tok0;       // equal shares: the cluster's first token
  int ntok;       // tokens of this cluster (with equal shares the first and last may be partial)
  int total;      // key tiles of this cluster, one stream across its tokens
  uint64_t wait_ns;
  volatile uint32_t* abort;
  __device__ uint32_t bar(int i) const { return sbase + kOffBars + 8 * i; }
};

// Entry modes of the kernel: the token's top-k list (kModeLists, whole tokens
// per cluster; kModeListsCut, equal shares of tiles), a sliding window of
// positions (kModeWindow), or a window followed by compressed-cache entries
// (kModeCompressed).  A compressed entry carries kCmpFlag through the index
// and row rings.
constexpr int kModeLists = 0;
constexpr int kModeWindow = 1;
constexpr int kModeCompressed = 2;
constexpr int kModeListsCut = 3;
constexpr int kCmpFlag = 1 << 30;
__host__ __device__ constexpr bool lists_mode(int mode) { return mode == kModeLists || mode == kModeListsCut; }

// Token of the m-th tile group of this cluster's stream.
template <int kMode>
__device__ __forceinline__ int token_of(const Params& p, const Ctx& c, int m) {
  if constexpr (kMode == kModeListsCut) return c.tok0 + m;
  else return c.cid + m * p.n_clusters;
}
// Token of stream position jj, and the position's tile within that token.
template <int kMode>
__device__ __forceinline__ int token_at(const Params& p, const Ctx& c, int jj) {
  if constexpr (kMode == kModeListsCut) return (c.first + jj) / p.n_tiles;
  else return c.cid + (jj / p.n_tiles) * p.n_clusters;
}
template <int kMode>
__device__ __forceinline__ int tile_at(const Params& p, const Ctx& c, int jj, int t) {
  if constexpr (kMode == kModeListsCut) return c.first + jj - t * p.n_tiles;
  else return jj % p.n_tiles;
}
// Stream positions [begin, end) of the cluster's m-th token.
template <int kMode>
__device__ __forceinline__ int seg_begin(const Params& p, const Ctx& c, int m) {
  if constexpr (kMode == kModeListsCut) return max((c.tok0 + m) * p.n_tiles, c.first) - c.first;
  else return m * p.n_tiles;
}
template <int kMode>
__device__ __forceinline__ int seg_end(const Params& p, const Ctx& c, int m) {
  if constexpr (kMode == kModeListsCut) return min((c.tok0 + m + 1) * p.n_tiles, c.first + c.total) - c.first;
  else return (m + 1) * p.n_tiles;
}
// Equal shares: first tile of cluster cl, and the cluster whose range holds
// tile g (the largest cl with start(cl) <= g).
__device__ __forceinline__ int cluster_start(const Params& p, int cl) {
  return static_cast<int>(static_cast<int64_t>(cl) * (p.T * p.n_tiles) / p.n_clusters);
}
__device__ __forceinline__ int cluster_of_tile(const Params& p, int g) {
  const int64_t tiles = p.T * p.n_tiles;
  return static_cast<int>((static_cast<int64_t>(g + 1) * p.n_clusters + tiles - 1) / tiles - 1);
}

__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity) {
  return mbar_wait<false>(c.bar(idx), parity, c.abort, c.wait_ns);
}
// Warp-uniform waits: every lane waits (bounded) and the warp agrees on the
// outcome, so warp-collective instructions after it never see a partial warp.
__device__ __forceinline__ bool warp_wait(const Ctx& c, int idx, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(c, idx, parity));
}
__device__ __forceinline__ bool warp_wait_cluster(const Ctx& c, int idx, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait<true>(c.bar(idx), parity, c.abort, c.wait_ns));
}

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void sts16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// 32-byte global store (both halves of a 64-byte-aligned pair of uint4 at p, p 32-byte aligned).
__device__ __forceinline__ void stg32(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
__device__ __forceinline__ int lds_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds16f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// Exchange layout of one column half (32 keys) of a partial score tile, in the
// staging and receive buffers: head h is a 128-byte row, 16-byte unit k (keys
// 4k .. 4k + 3 of the half) of row h at k ^ (h & 7), so a warp's 32 rows spread
// over all banks; the 32 rows of a TMEM lane quadrant form one 4 KB block.
__device__ __forceinline__ uint32_t xchg_offset(int h, int k) {
  return static_cast<uint32_t>(h * 128 + ((k ^ (h & 7)) << 4));
}

// ------------------------------------------------------------------ index warp
// Two index warps take alternate passes of kIdxBatch tiles (warp iw owns the
// ring slots [kIdxBatch iw, kIdxBatch iw + kIdxBatch)), so two chains of
// dependent loads (top-k entry, then block_table) are in flight at once.  Each
// warp loads the top-k entries of its next pass before it resolves the
// current one.
static_assert(kIdxBatch == 4, "two entries per lane per tile, four tiles per pass");

// Sequence of stream tile jj (jj < c.total).
template <int kMode>
__device__ __forceinline__ int seq_of_tile(const Params& p, const Ctx& c, int jj) {
  return token_at<kMode>(p, c, jj) / p.S1;
}

// Entries of the pass starting at stream tile j0, -1 beyond the stream or the
// list.  Lists: logical positions from topk_idx.  Window: the positions
// p - window + 1 + e of the token at p = act_seqs[b] - S1 + s (its sequence's
// newest S1 positions are the S1 query tokens; negative positions are -1).
// Compressed: the window, then entry e' = e - window is compressed entry
// e' (CFA) or cmp_idx[t, e'] (SCFA), kept when (i + 1) * cmp_ratio - 1 <= p:
// entry i summarises positions [i * r, (i + 1) * r) and exists from the
// position that completes it on.
template <int kMode>
__device__ __forceinline__ void index_load(const Params& p, const Ctx& c, int j0, int lane, int (&idx)[8]) {
#pragma unroll
  for (int k = 0; k < kIdxBatch; ++k) {
    const int jj = j0 + k;
    const int t = token_at<kMode>(p, c, jj);
    const int e0 = tile_at<kMode>(p, c, jj, t) * kTileKeys + lane;
    if constexpr (!lists_mode(kMode)) {
      const int b = t / p.S1;
      const int pos = (jj < c.total ? __ldg(p.act_seqs + b) : 0) - p.S1 + (t - b * p.S1);
      const int first = pos - p.window + 1;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + 32 * u;
        int v = -1;
        if (jj < c.total && e < p.topk) {
          if (e < p.window) {
            v = first + e >= 0 ? first + e : -1;
          } else if constexpr (kMode == kModeCompressed) {
            const int e2 = e - p.window;
            const int ci = p.cmp_idx != nullptr ? __ldg(p.cmp_idx + static_cast<int64_t>(t) * p.cmp_topk + e2) : e2;
            v = (ci >= 0 && ci < (1 << 29) && static_cast<int64_t>(ci + 1) * p.cmp_ratio - 1 <= pos) ? (ci | kCmpFlag)
                                                                                                   : -1;
          }
        }
        idx[2 * k + u] = v;
      }
    } else {
      const int32_t* tk = p.topk_idx + static_cast<int64_t>(t) * p.topk;
#pragma unroll
      for (int u = 0; u < 2; ++u)
        idx[2 * k + u] = (jj < c.total && e0 + 32 * u < p.topk) ? __ldg(tk + e0 + 32 * u) : -1;
    }
  }
}

// `idx` holds the entries of this warp's first pass, loaded before the CTA's
// set-up barrier.  The stream runs through the cluster's tokens in order; a
// pass may straddle two tokens, so each tile's sequence is found from its
// position in the stream.
template <int kMode>
__device__ void index_role(const Params& p, const Ctx& c, int iw, int lane, int (&idx)[8]) {
  int32_t* rows = reinterpret_cast<int32_t*>(c.smem + kOffRows);
  // pull the cluster's top-k rows and their sequences' block-table rows towards
  // L2 up front (one 128-byte line per prefetch; the warps split the lines)
  for (int m = 0; m < c.ntok; ++m) {
    const int t = token_of<kMode>(p, c, m);
    const int32_t* bt = p.block_table + static_cast<int64_t>(t / p.S1) * p.mbps;
    if constexpr (lists_mode(kMode)) {  // only list modes read topk_idx
      const int32_t* tk = p.topk_idx + static_cast<int64_t>(t) * p.topk;
      for (int e = (iw * 32 + lane) * 32; e < p.topk + 32; e += kIndexWarps * 32 * 32)
        prefetch_l2(tk + min(e, p.topk - 1));
    }
    for (int e = (iw * 32 + lane) * 32; e < p.mbps + 32; e += kIndexWarps * 32 * 32) prefetch_l2(bt + min(e, p.mbps - 1));
  }
  bool bad = false;
  for (int j0 = iw * kIdxBatch; j0 < c.total; j0 += kIndexWarps * kIdxBatch) {
    const int nb = min(kIdxBatch, c.total - j0);
    int blk[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      // the table entry is loaded for any index inside the table (without
      // waiting for the length check); entries outside [0, act) are dropped below
      if constexpr (kMode == kModeCompressed) {
        const bool cmp = idx[q] >= 0 && (idx[q] & kCmpFlag);
        const int slot = (idx[q] & ~kCmpFlag) >> 7;
        const int mb = cmp ? p.cmp_mbps : p.mbps;
        const int32_t* bt = cmp ? p.cmp_block_table : p.block_table;
        blk[q] = (idx[q] >= 0 && slot < mb)
                     ? __ldg(bt + static_cast<int64_t>(seq_of_tile<kMode>(p, c, j0 + (q >> 1))) * mb + slot)
                     : -1;
      } else {
        const int slot = idx[q] >> 7;
        blk[q] = (idx[q] >= 0 && slot < p.mbps)
                     ? __ldg(p.block_table + static_cast<int64_t>(seq_of_tile<kMode>(p, c, j0 + (q >> 1))) * p.mbps + slot)
                     : -1;
      }
    }
    // the sequence lengths too, so that their latency overlaps the table loads
    int act[kIdxBatch];
#pragma unroll
    for (int k = 0; k < kIdxBatch; ++k) act[k] = k < nb ? __ldg(p.act_seqs + seq_of_tile<kMode>(p, c, j0 + k)) : 0;
    int nxt[8];
    index_load<kMode>(p, c, j0 + kIndexWarps * kIdxBatch, lane, nxt);
    bool ok = true;
    for (int k = 0; k < nb && ok; ++k) {
      const int j = j0 + k;
      ok = warp_wait(c, kBarIdxEmpty + (j % kIdxSlots), ((j / kIdxSlots) & 1) ^ 1);
    }
    if (!ok) break;
#pragma unroll
    for (int k = 0; k < kIdxBatch; ++k) {
      if (k >= nb) continue;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = 2 * k + u;
        // a compressed entry was checked for visibility when it was loaded
        const bool cmp = kMode == kModeCompressed && idx[q] >= 0 && (idx[q] & kCmpFlag);
        const bool in_seq = idx[q] >= 0 && (cmp || idx[q] < act[k]);
        const bool valid = in_seq && blk[q] >= 0 && blk[q] < (cmp ? p.cmp_num_blocks : p.num_blocks);
        if (in_seq && !valid) bad = true;
        const int row = (blk[q] * 128 + (idx[q] & 127)) | (cmp ? kCmpFlag : 0);
        rows[((j0 + k) % kIdxSlots) * kTileKeys + u * 32 + lane] = valid ? row : -1;
      }
    }
    for (int k = 0; k < nb; ++k) mbar_arrive(c.bar(kBarIdxFull + ((j0 + k) % kIdxSlots)));
#pragma unroll
    for (int q = 0; q < 8; ++q) idx[q] = nxt[q];
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&g_mla_status, MLA_DEVICE_BAD_BLOCK);
}

// ------------------------------------------------------------------ gather warps
// Stage layout (per 64-key tile): chunks 0-3 hold this CTA's latent dims
// [64c, 64c+64) in 128-byte rows (unit u of key k at u ^ (k & 7)); the rope
// chunk holds this CTA's 32 rope dims in 64-byte rows (unit u of key k at
// u ^ ((k >> 1) & 3)).
__device__ __forceinline__ uint32_t rope_unit(int k, int u) {
  return static_cast<uint32_t>(k * 64 + ((u ^ ((k >> 1) & 3)) << 4));
}

// INT8 path: "INT8 quantization path" -- INT8 -> FP16 -> FP32 (exact), times
// the group scale (one fp32 rounding), -> BF16.
__device__ __forceinline__ void dequant4(uint32_t w, float s, uint32_t& lo, uint32_t& hi) {
  const float f0 = __fmul_rn(__int2float_rn(static_cast<int>(w << 24) >> 24), s);
  const float f1 = __fmul_rn(__int2float_rn(static_cast<int>(w << 16) >> 24), s);
  const float f2 = __fmul_rn(__int2float_rn(static_cast<int>(w << 8) >> 24), s);
  const float f3 = __fmul_rn(__int2float_rn(static_cast<int>(w) >> 24), s);
  lo = pack_bf16x2(f0, f1);
  hi = pack_bf16x2(f2, f3);
}

// Row of the original or (mode 2, kCmpFlag) the compressed cache: base
// pointer and row index for a valid ring entry.
template <int kMode>
__device__ __forceinline__ const uint8_t* row_base(const uint8_t* ori, const uint8_t* cmp, int32_t row, int64_t bytes) {
  if constexpr (kMode == kModeCompressed) {
    if (row & kCmpFlag) return cmp + static_cast<int64_t>(row & ~kCmpFlag) * bytes;
  }
  return ori + static_cast<int64_t>(row) * bytes;
}

template <bool kInt8, int kMode>
__device__ void gather_role(const Params& p, const Ctx& c, int gw, int lane) {
  // all eight warps work on every tile; warp gw takes keys [8 gw, 8 gw + 8)
  const int key0 = gw * 8;
  const int32_t* rows_all = reinterpret_cast<const int32_t*>(c.smem + kOffRows);
  uint8_t* vmask8 = c.smem + kOffVmask;
  const uint8_t* kvr = reinterpret_cast<const uint8_t*>(p.kv_rope) + c.crank * 64 + (lane & 3) * 16;
  const uint8_t* cmr = reinterpret_cast<const uint8_t*>(p.cmp_rope) + c.crank * 64 + (lane & 3) * 16;
  const int rk = key0 + (lane >> 2);  // rope: four 16-byte units per key, one per lane
  for (int j = 0; j < c.total; ++j) {
    const int st = j % kStages;
    const int slot = j % kIdxSlots;
    if (!warp_wait(c, kBarEmpty + st, ((j / kStages) & 1) ^ 1)) break;
    if (!warp_wait(c, kBarIdxFull + slot, (j / kIdxSlots) & 1)) break;
    const int32_t* rows = rows_all + slot * kTileKeys;
    const uint32_t vbits = __ballot_sync(0xffffffffu, lane < 8 && rows[key0 + (lane & 7)] >= 0) & 0xFFu;
    const int32_t rr = rows[rk];
    const uint32_t stage = c.sbase + kOffStages + st * kStageBytes;
    const uint32_t rope = stage + 4 * kChunkBytes;
    if constexpr (!kInt8) {
      // latent half: 512 B per key, one key per warp instruction (32 lanes x 16 B)
      const uint8_t* kvn = reinterpret_cast<const uint8_t*>(p.kv_nope) + c.crank * 512 + lane * 16;
      const uint8_t* cmn = reinterpret_cast<const uint8_t*>(p.cmp_nope) + c.crank * 512 + lane * 16;
      const uint32_t chunk = stage + (lane >> 3) * kChunkBytes;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int key = key0 + i;
        const int32_t row = rows[key];
        cp_async_16(chunk + key * 128 + (((lane & 7) ^ (key & 7)) << 4),
                    row >= 0 ? row_base<kMode>(kvn, cmn, row, 1024) : kvn, row >= 0 ? 16u : 0u);
      }
      cp_async_16(rope + rope_unit(rk, lane & 3), rr >= 0 ? row_base<kMode>(kvr, cmr, rr, 128) : kvr,
                  rr >= 0 ? 16u : 0u);
      mbar_arrive_relaxed(c.bar(kBarIdxEmpty + slot));
      cp_async_arrive_noinc(c.bar(kBarFull + st));
      if (lane == 0) {
        vmask8[st * 8 + gw] = static_cast<uint8_t>(vbits);
        mbar_arrive(c.bar(kBarFull + st));  // releases the mask byte
      }
    } else {
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      // latent half: 256 int8 per key = 16 lanes x 16 B; lanes 16-31 take the next key
      const int u = lane & 15;
      const uint8_t* kvn = reinterpret_cast<const uint8_t*>(p.kv_nope) + c.crank * 256 + u * 16;
      const uint8_t* cmn = reinterpret_cast<const uint8_t*>(p.cmp_nope) + c.crank * 256 + u * 16;
      const uint8_t* scl = reinterpret_cast<const uint8_t*>(p.kv_scales + c.crank * 2 + (u >> 3));
      const uint8_t* cms = reinterpret_cast<const uint8_t*>(p.cmp_scales + c.crank * 2 + (u >> 3));
      uint4 v[4];
      float sc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t row = rows[key0 + 2 * i + (lane >> 4)];
        v[i] = row >= 0 ? ldg16(row_base<kMode>(kvn, cmn, row, 512)) : zero;
        sc[i] = row >= 0 ? __ldg(reinterpret_cast<const float*>(row_base<kMode>(scl, cms, row, 16))) : 0.f;
      }
      const uint4 qr = rr >= 0 ? ldg16(row_base<kMode>(kvr, cmr, rr, 128)) : zero;
      mbar_arrive_relaxed(c.bar(kBarIdxEmpty + slot));
      const uint32_t chunk = stage + (u >> 2) * kChunkBytes;
      const int u8 = (u & 3) * 2;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = key0 + 2 * i + (lane >> 4);
        uint4 a, b2;
        dequant4(v[i].x, sc[i], a.x, a.y);
        dequant4(v[i].y, sc[i], a.z, a.w);
        dequant4(v[i].z, sc[i], b2.x, b2.y);
        dequant4(v[i].w, sc[i], b2.z, b2.w);
        sts16(chunk + key * 128 + ((u8 ^ (key & 7)) << 4), a);
        sts16(chunk + key * 128 + (((u8 + 1) ^ (key & 7)) << 4), b2);
      }
      sts16(rope + rope_unit(rk, lane & 3), qr);
      if (lane == 0) vmask8[st * 8 + gw] = static_cast<uint8_t>(vbits);
      fence_proxy_async_smem();
      mbar_arrive(c.bar(kBarFull + st));
    }
  }
  cp_async_wait_all();  // no copy of this thread lands after the CTA has left its roles
}

// ------------------------------------------------------------------ sender warps
// Copy the CTA's partial score tile (128 heads x 64 keys, fp32) into the
// peer's receive slots, one column half at a time: TMEM -> registers -> the
// local staging buffer, then bulk copies by the TMA engine, so the CTA-to-CTA
// traffic never queues in front of the softmax warps' shared-memory accesses.
// Column half c of tile j goes to slot c once the peer has read half c of
// tile j - 1 out of it.
__device__ __forceinline__ bool send_half(const Ctx& c, const uint32_t (&v)[32], int h, int q, int lane, int j,
                                          int half, uint32_t stg, uint32_t dst, uint32_t rbar) {
  // this half's previous copy has left its staging buffer (the other half's
  // most recent copy may still be reading its own)
  if (lane == 0) bulk_wait_read_but_one();
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) sts16(stg + xchg_offset(h, k), make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
  fence_proxy_async_smem();  // generic-proxy stores -> bulk-copy reads
  __syncwarp();
  bool ok = true;
  if (lane == 0) {
    if (j > 0) ok = mbar_wait<true>(c.bar(kBarPeerFree + half), (j - 1) & 1, c.abort, c.wait_ns);
    if (ok) {
      const uint32_t blk = static_cast<uint32_t>(q) * kXchgBlockBytes;
      bulk_copy_to_peer(dst + blk, stg + blk, kXchgBlockBytes, rbar);
      bulk_commit();
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Exchange 32-byte pieces among each group of four lanes so that lane l of
// the group ends with piece l of the group's e-th line in v[2 e], v[2 e + 1]
// (two butterfly stages; the same call undoes it).  v holds four 32-byte
// pieces (eight uint4) per lane.
__device__ __forceinline__ void transpose4x32(uint4 (&v)[8], int lane) {
  const int l4 = lane & 3;
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {
    const bool b = (l4 & bit) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (e & bit) continue;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint4& lo = v[2 * e + u];
        uint4& hi = v[2 * (e + bit) + u];
        const uint4 snd = b ? lo : hi;
        uint4 rcv;
        rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, bit);
        rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, bit);
        rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, bit);
        rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, bit);
        if (b) lo = rcv; else hi = rcv;
      }
    }
  }
}

// The shared-memory part of one token's Q for the 32 heads of TMEM lane
// quadrant q (qn0, qr0: the quadrant's first head row, this CTA's dims):
// latent dims [128, 256) as 128-byte swizzled rows of 64 dims (head h at row
// h of chunk (d - 128) / 64) and the 32 rope dims, by cp.async, zero-filled
// for heads beyond n_q.  Lanes take whole 128-byte lines, not heads: the
// heads' rows lie 1 KB apart, so a warp-wide copy covers 4 lines (rope: 8
// half lines) instead of 32 pieces.
__device__ __forceinline__ void copy_q_smem(const Params& p, const Ctx& c, int q, int lane, const uint8_t* qn0,
                                            const uint8_t* qr0) {
  // dims [128, 256): line L = 4 i + lane / 8 of the warp's 64 (head L / 2, chunk L % 2), unit lane % 8
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int L = 4 * i + (lane >> 3), hh = L >> 1, ch = L & 1, u = lane & 7;
    const int h = q * 32 + hh;
    const bool live = h < p.n_q;
    cp_async_16(c.sbase + kOffQHalf + ch * (kQHalfBytes / 2) + h * 128 + ((u ^ (h & 7)) << 4),
                live ? static_cast<const void*>(qn0 + static_cast<int64_t>(hh) * 1024 + 256 + ch * 128 + u * 16)
                     : p.q_nope,
                live ? 16u : 0u);
  }
  // rope: head 8 i + lane / 4, unit lane % 4
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int hh = 8 * i + (lane >> 2), u = lane & 3;
    const int h = q * 32 + hh;
    const bool live = h < p.n_q;
    cp_async_16(c.sbase + kOffQRope + rope_unit(h, u),
                live ? static_cast<const void*>(qr0 + static_cast<int64_t>(hh) * 128 + u * 16) : p.q_rope,
                live ? 16u : 0u);
  }
}

// Q of one token for sender warp q (heads [32 q, 32 q + 32), rows qrow0 ..
// qrow0 + 31): the CTA's latent dims [128, 256) (128-byte swizzled rows of 64
// dims, head h at row h of chunk (d - 128) / 64) and its 32 rope dims go to
// shared memory by cp.async (zero-filled for heads beyond n_q), then dims
// [0, 128) to TMEM (the lanes of the quadrant) through registers; then
// QReady.  The heads' rows lie 1 KB apart, so the copies for shared memory
// assign lanes to whole 128-byte lines rather than to heads (a warp-wide copy
// then covers 4 lines, not 32).  In the window modes the TMEM dims land the
// same way in the warp's two staging blocks (idle between a token's last
// partial tile and the next token's first) and are read back per head; the
// list modes load them per head.  The senders load
// each token's Q as soon as the previous token's score MMAs are complete, so
// the load overlaps the softmax of that token's last tiles.
template <int kMode>
__device__ __forceinline__ void load_q(const Params& p, const Ctx& c, int q, int lane, int64_t qrow0, uint32_t tQ) {
  const uint8_t* qn0 = reinterpret_cast<const uint8_t*>(p.q_nope) + (qrow0 * 512 + c.crank * 256) * 2;
  const uint8_t* qr0 = reinterpret_cast<const uint8_t*>(p.q_rope) + (qrow0 * 64 + c.crank * 32) * 2;
  copy_q_smem(p, c, q, lane, qn0, qr0);
  if constexpr (!lists_mode(kMode)) {
    // Window modes (a token switch every few tiles): dims [0, 128) by
    // line-major copies into this warp's two 4 KB staging blocks (line ch of
    // head hh at block ch, row hh, 16-byte unit u at u ^ (hh & 7)), read back
    // per head once the blocks' last bulk copies to the peer have read them
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    const uint32_t blk[2] = {c.sbase + kOffStaging + q * kXchgBlockBytes,
                             c.sbase + kOffStaging + kXchgBytes + q * kXchgBlockBytes};
    {
      // lane: line chunk (lane / 8) % 2 and unit lane % 8 of heads 2 i + lane / 16
      const int ch = (lane >> 3) & 1, u = lane & 7, h0 = lane >> 4;
      const uint8_t* src = qn0 + static_cast<int64_t>(h0) * 1024 + ch * 128 + u * 16;
      const uint32_t dst = (ch ? blk[1] : blk[0]) + h0 * 128;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int hh = 2 * i + h0;
        const bool live = q * 32 + hh < p.n_q;
        cp_async_16(dst + i * 256 + ((u ^ (hh & 7)) << 4), live ? static_cast<const void*>(src + i * 2048) : p.q_nope,
                    live ? 16u : 0u);
      }
    }
    cp_async_wait_all();
    __syncwarp();  // every lane's copies have landed before any lane reads another's
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t w[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 v = lds16f(blk[ch] + lane * 128 + ((u ^ (lane & 7)) << 4));
        w[4 * u + 0] = __float_as_uint(v.x);
        w[4 * u + 1] = __float_as_uint(v.y);
        w[4 * u + 2] = __float_as_uint(v.z);
        w[4 * u + 3] = __float_as_uint(v.w);
      }
      tmem_st_32x32b_x32(tQ + 32 * ch, w);
    }
    __syncwarp();  // the staging blocks are read before the next partial tile is staged
  } else {
    // top-k lists (a switch every 32 tiles): per head into registers, which
    // keeps the senders' per-tile code free of spills
    const bool live = q * 32 + lane < p.n_q;
    const uint8_t* qn = qn0 + static_cast<int64_t>(lane) * 1024;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 qv[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) qv[u] = live ? ldg16(qn + u * 16) : zero;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t w[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        w[4 * u + 0] = qv[8 * ch + u].x;
        w[4 * u + 1] = qv[8 * ch + u].y;
        w[4 * u + 2] = qv[8 * ch + u].z;
        w[4 * u + 3] = qv[8 * ch + u].w;
      }
      tmem_st_32x32b_x32(tQ + 32 * ch, w);
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();  // cp.async data -> tensor-core reads
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(c.bar(kBarQReady));
}

template <bool kInt8, int kMode>
__device__ void sender_role(const Params& p, const Ctx& c, int q, int lane) {
  const int h = q * 32 + lane;
  const uint32_t tQ = c.tmem + (static_cast<uint32_t>(q * 32) << 16) + kTmemQ;
  const uint32_t tR = c.tmem + (static_cast<uint32_t>(q * 32) << 16) + kTmemRegion;
  const uint32_t peer = c.crank ^ 1u;
  const uint32_t stg = c.sbase + kOffStaging;
  const uint32_t dst = mapa_shared(c.sbase + kOffRecv, peer);
  const uint32_t rbar0 = mapa_shared(c.bar(kBarRecvFull + 0), peer);
  const uint32_t rbar1 = mapa_shared(c.bar(kBarRecvFull + 1), peer);
  if constexpr (!kInt8) load_q<kMode>(p, c, q, lane, static_cast<int64_t>(token_of<kMode>(p, c, 0)) * p.n_q + q * 32, tQ);
  int m = 0, m_end = seg_end<kMode>(p, c, 0);  // token ordinal and the end of its segment
  // the loop bound comes from shared memory: the two 32-column halves held in
  // registers leave none to spare for it
  for (int j = 0; j < lds_s32(c.sbase + kOffTotal); ++j) {
    const int r = j % kRegions;
    if (!warp_wait(c, kBarSFull + r, (j / kRegions) & 1)) break;
    tc_fence_after();
    uint32_t a[32], b[32];
    tmem_ld_32x32b_x32(tR + 64 * r, a);
    tmem_ld_32x32b_x32(tR + 64 * r + 32, b);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive_relaxed(c.bar(kBarSFree + r));  // the values are in registers (wait::ld)
    if (!send_half(c, a, h, q, lane, j, 0, stg, dst, rbar0)) break;
    if (!send_half(c, b, h, q, lane, j, 1, stg + kXchgBytes, dst + kXchgBytes, rbar1)) break;
    if (!kInt8 && j + 1 == m_end && m + 1 < c.ntok) {
      // the next token's Q replaces this one's once its score MMAs are complete
      if (!warp_wait(c, kBarQFree, m & 1)) break;
      tc_fence_after();
      ++m;
      load_q<kMode>(p, c, q, lane, static_cast<int64_t>(token_of<kMode>(p, c, m)) * p.n_q + q * 32, tQ);
      m_end = seg_end<kMode>(p, c, m);
    }
  }
  // the peer cannot leave before this CTA reaches its final cluster barrier,
  // which waits for these copies to complete
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

// ------------------------------------------------------------------ MMA warp
__device__ __forceinline__ void issue_s(const Ctx& c, int k) {
  constexpr uint32_t idesc = make_idesc_f16(128, 64, 1, 0, 0);
  const uint32_t qrope = c.sbase + kOffQRope;
  const uint32_t qhalf = c.sbase + kOffQHalf;
  const uint32_t stage = c.sbase + kOffStages + (k % kStages) * kStageBytes;
  fence_proxy_async_smem();  // cp.async / st.shared data -> tensor-core reads
  tc_fence_after();
  // S = Q_latent K_latent^T (dims [0, 128): A = Q in TMEM; dims [128, 256): A = Q
  // in smem) + Q_rope K_rope^T (A = Q rope in smem)
  const uint32_t dS = c.tmem + kTmemRegion + 64 * (k % kRegions);
#pragma unroll
  for (int s = 0; s < 8; ++s)
    umma_ts(dS, c.tmem + kTmemQ + 8 * s,
            make_sdesc(stage + (s >> 2) * kChunkBytes + (s & 3) * 32, 16, 1024, kSwizzle128B), idesc, s > 0 ? 1u : 0u);
#pragma unroll
  for (int s = 8; s < 16; ++s)
    umma_ss(dS, make_sdesc(qhalf + ((s - 8) >> 2) * (kQHalfBytes / 2) + ((s - 8) & 3) * 32, 16, 1024, kSwizzle128B),
            make_sdesc(stage + (s >> 2) * kChunkBytes + (s & 3) * 32, 16, 1024, kSwizzle128B), idesc, 1u);
#pragma unroll
  for (int s = 0; s < 2; ++s)
    umma_ss(dS, make_sdesc(qrope + s * 32, 16, 512, kSwizzle64B),
            make_sdesc(stage + 4 * kChunkBytes + s * 32, 16, 512, kSwizzle64B), idesc, 1u);
  umma_commit(c.bar(kBarSFull + k % kRegions));
}

__device__ __forceinline__ void issue_pv(const Ctx& c, int i, bool first_of_token) {
  constexpr uint32_t idesc = make_idesc_f16(128, 256, 1, 0, 1);
  const uint32_t stage = c.sbase + kOffStages + (i % kStages) * kStageBytes;
  const uint32_t aP = c.tmem + kTmemRegion + 64 * (i % kRegions);
  tc_fence_after();
  // O += P_hi . V, then O += P_lo . V (same V tile, 16 keys per instruction)
#pragma unroll
  for (int s = 0; s < 8; ++s)
    umma_ts(c.tmem + kTmemO, aP + (s < 4 ? 0 : 32) + 8 * (s & 3),
            make_sdesc(stage + (s & 3) * 16 * 128, kChunkBytes, 1024, kSwizzle128B), idesc,
            (!first_of_token || s > 0) ? 1u : 0u);
  umma_commit(c.bar(kBarPvDone + i % kRegions));
  umma_commit(c.bar(kBarEmpty + (i % kStages)));
}

// One thread polls both hand-offs and issues whichever is ready: P.V(kp) as
// soon as the softmax has written P(kp), and S(ks) once its key tile has
// landed and P.V(ks - 3) has released TMEM region ks % 3, so a stage is
// released as early as the data allows and the softmax of one tile overlaps
// with the P.V of the previous one.  The stream runs through the cluster's
// tokens: the first S of token m also waits for its Q (QReady phase m), the
// last S of a token is followed by a commit to QFree (its Q may then be
// replaced), and the first P.V of token m > 0 waits until O of token m - 1 has
// been read out (OFree phase m - 1) and starts a fresh accumulator.
template <int kMode>
__device__ void mma_role(const Params& p, const Ctx& c) {
  bool ok = true;
  int ks = 0, kp = 0;
  int s_tok = 0, s_in = 0;  // token ordinal and tile-in-segment of ks
  int p_tok = 0, p_in = 0;  // the same for kp
  int s_len = seg_end<kMode>(p, c, 0) - seg_begin<kMode>(p, c, 0), p_len = s_len;  // tiles of the token's segment
  bool s_q = false;         // Q of token s_tok seen ready
  uint64_t t_idle = 0;
  uint32_t spins = 0;
  while (ok && kp < c.total) {
    bool progressed = false;
    if (kp < ks && mbar_poll(c.bar(kBarPFull + kp % kRegions), (kp / kRegions) & 1) &&
        (p_in != 0 || p_tok == 0 || mbar_poll(c.bar(kBarOFree), (p_tok - 1) & 1))) {
      issue_pv(c, kp, p_in == 0);
      ++kp;
      if (++p_in == p_len) {
        p_in = 0;
        ++p_tok;
        p_len = seg_end<kMode>(p, c, p_tok) - seg_begin<kMode>(p, c, p_tok);
      }
      progressed = true;
    }
    if (ks < c.total) {
      if (!s_q) s_q = mbar_poll(c.bar(kBarQReady), s_tok & 1);
      if (s_q && mbar_poll(c.bar(kBarFull + ks % kStages), (ks / kStages) & 1) &&
          (ks < kRegions || mbar_poll(c.bar(kBarPvDone + ks % kRegions), ((ks / kRegions) & 1) ^ 1))) {
        issue_s(c, ks);
        ++ks;
        if (++s_in == s_len) {
          umma_commit(c.bar(kBarQFree));  // the token's score MMAs: its Q may be replaced
          s_in = 0;
          ++s_tok;
          s_len = seg_end<kMode>(p, c, s_tok) - seg_begin<kMode>(p, c, s_tok);
          s_q = false;
        }
        progressed = true;
      }
    }
    if (progressed) {
      spins = 0;
    } else if ((++spins & 255u) == 0) {
      // bounded like every other wait: give up after the limit without progress
      const uint64_t now = globaltimer_ns();
      if (t_idle == 0 || spins == 256u) t_idle = now;
      if (*c.abort) ok = false;
      else if (now - t_idle > c.wait_ns) { *c.abort = 1u; ok = false; }
    }
  }
  umma_commit(c.bar(kBarFinal));
  volatile uint32_t never = 0;
  mbar_wait<false>(c.bar(kBarFinal), 0, &never, c.wait_ns > 500000000ull ? c.wait_ns : 500000000ull);
}

// ------------------------------------------------------------------ softmax warps
// INT8 instantiations: Q of token qrow / n_q loaded by the softmax warps
// (measured faster there than on the senders, whose registers the INT8
// kernels cannot spare).  Warps of column half 0 put the CTA's latent dims
// [0, 128) of their heads into TMEM (loaded line-major by groups of four
// lanes, transposed back to one head per lane); warps of column half 1 copy their
// quadrant's latent dims [128, 256) and all four rope units into shared
// memory by cp.async, lanes assigned to whole 128-byte lines (the heads' rows
// lie 1 KB apart); then QReady.
__device__ __forceinline__ void load_q_softmax(const Params& p, const Ctx& c, int h, int half, bool live,
                                               int64_t qrow, uint32_t tQ) {
  const int lane = h & 31, q = h >> 5;
  if (half == 0) {
    // latent dims [0, 128): loaded line-major (32-byte piece lane % 4 of each
    // line of the four-lane group's heads), then transposed back to one head
    // per lane; all loads are issued before the first TMEM store (inline asm
    // that may touch memory would otherwise hold back every later load)
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t qrow0 = qrow - lane;
    const uint8_t* qn0 = reinterpret_cast<const uint8_t*>(p.q_nope) + (qrow0 * 512 + c.crank * 256) * 2;
    const int g4 = lane & ~3, l4 = lane & 3;
    uint4 qv[2][8];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool hlive = q * 32 + g4 + e < p.n_q;
        const uint8_t* src = qn0 + static_cast<int64_t>(g4 + e) * 1024 + ch * 128 + l4 * 32;
        qv[ch][2 * e] = hlive ? ldg16(src) : zero;
        qv[ch][2 * e + 1] = hlive ? ldg16(src + 16) : zero;
      }
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      transpose4x32(qv[ch], lane);
      uint32_t w[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        w[4 * u + 0] = qv[ch][u].x;
        w[4 * u + 1] = qv[ch][u].y;
        w[4 * u + 2] = qv[ch][u].z;
        w[4 * u + 3] = qv[ch][u].w;
      }
      tmem_st_32x32b_x32(tQ + 32 * ch, w);
    }
  } else {
    const int64_t qrow0 = qrow - lane;
    copy_q_smem(p, c, q, lane, reinterpret_cast<const uint8_t*>(p.q_nope) + (qrow0 * 512 + c.crank * 256) * 2,
                reinterpret_cast<const uint8_t*>(p.q_rope) + (qrow0 * 64 + c.crank * 32) * 2);
  }
  cp_async_wait_all();
  fence_proxy_async_smem();  // cp.async data -> tensor-core reads
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(c.bar(kBarQReady));
}

// ------------------------------------------------------------------ cut tokens
// With equal shares, a token's tiles may be cut between consecutive clusters.
// Each part ends with its own online softmax state: O relative to its running
// max m (log2 units) and its row sum l.  The parts combine exactly as in the
// flash update: with M = max m_k and w_k = 2^(m_k - M),
// O = sum w_k O_k / sum w_k l_k and lse = M + log2(sum w_k l_k).

// Slot of the part of token t computed by cluster cl, CTA rank r: segment 0
// holds the cluster's first token, segment 1 its last (a cut token is one of
// the two).
__device__ __forceinline__ float* part_slot(const Params& p, int cl, int t, uint32_t r) {
  const int seg = t == cluster_start(p, cl) / p.n_tiles ? 0 : 1;
  return p.ws + (static_cast<int64_t>(cl * 2 + seg) * 2 + r) * kSlotFloats;
}

// Store this cluster's part of cut token t (O in TMEM at tO, m, l_tot), then
// release O for the next token.  The TMEM loads are warp-wide; only live
// heads store.
__device__ __noinline__ void store_part(const Params& p, const Ctx& c, int t, int h, int half, bool live, uint32_t tO,
                                        float m, float l_tot) {
  float* own = part_slot(p, c.cid, t, c.crank);
  float4* so = reinterpret_cast<float4*>(own) + half * 32 * kHeads + h;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + 32 * ch, o);
    tmem_wait_ld();
    if (live) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        so[(ch * 8 + k) * kHeads] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
    }
  }
  if (live && half == 0) {
    own[kHeads * 256 + h] = m;
    own[kHeads * 256 + kHeads + h] = l_tot;
  }
  tc_fence_before();
  mbar_arrive(c.bar(kBarOFree));
}

// One block per (token, CTA rank, 8 of the rank's 256 latent dims), one thread
// per head: merges the parts of a cut token in one pass, with the running
// maximum of the flash update (tokens that are not cut return at once).  The
// parts are read eight at a time so that their loads are in flight together.
// Runs after the attention kernel on the same stream.
constexpr int kCombineDims = 8;
constexpr int kCombineParts = 8;
__global__ void __launch_bounds__(kHeads) combine_kernel(const __grid_constant__ Params p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the attention kernel's stores are visible
  const int t = blockIdx.x, r = blockIdx.y, ch = blockIdx.z, h = threadIdx.x;
  const int g0 = t * p.n_tiles;
  const int c_first = cluster_of_tile(p, g0), c_last = cluster_of_tile(p, g0 + p.n_tiles - 1);
  if (c_first == c_last || h >= p.n_q) return;
  // dims [8 ch, 8 ch + 8) of the rank: column half ch / 16, float4 units (ch % 16) * 2 + {0, 1}
  const int unit0 = ((ch >> 4) * 32 + (ch & 15) * 2) * kHeads + h;
  float mx = -INFINITY, lsum = 0.f, acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  for (int base = c_first; base <= c_last; base += kCombineParts) {
    float mk[kCombineParts], lk[kCombineParts];
    float4 v[kCombineParts][2];
#pragma unroll
    for (int u = 0; u < kCombineParts; ++u) {
      const bool in = base + u <= c_last;
      const float* sl = part_slot(p, in ? base + u : c_last, t, r);
      mk[u] = in ? __ldcg(sl + kHeads * 256 + h) : -INFINITY;
      lk[u] = in ? __ldcg(sl + kHeads * 256 + kHeads + h) : 0.f;
      const float4* src = reinterpret_cast<const float4*>(sl) + unit0;
      v[u][0] = in ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[u][1] = in ? __ldcg(src + kHeads) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kCombineParts; ++u) {
      if (mk[u] == -INFINITY) continue;  // a part without a valid key adds nothing
      if (mk[u] > mx) {
        const float f = mx == -INFINITY ? 0.f : exp2f(mx - mk[u]);
        lsum *= f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] *= f;
        mx = mk[u];
      }
      const float w = exp2f(mk[u] - mx);
      lsum = fmaf(w, lk[u], lsum);
      acc[0] = fmaf(w, v[u][0].x, acc[0]);
      acc[1] = fmaf(w, v[u][0].y, acc[1]);
      acc[2] = fmaf(w, v[u][0].z, acc[2]);
      acc[3] = fmaf(w, v[u][0].w, acc[3]);
      acc[4] = fmaf(w, v[u][1].x, acc[4]);
      acc[5] = fmaf(w, v[u][1].y, acc[5]);
      acc[6] = fmaf(w, v[u][1].z, acc[6]);
      acc[7] = fmaf(w, v[u][1].w, acc[7]);
    }
  }
  const float inv_l = lsum > 0.f ? 1.f / lsum : 0.f;
  const int64_t qrow = static_cast<int64_t>(t) * p.n_q + h;
  *reinterpret_cast<uint4*>(p.out + qrow * 512 + r * 256 + ch * kCombineDims) =
      make_uint4(pack_bf16x2(acc[0] * inv_l, acc[1] * inv_l), pack_bf16x2(acc[2] * inv_l, acc[3] * inv_l),
                 pack_bf16x2(acc[4] * inv_l, acc[5] * inv_l), pack_bf16x2(acc[6] * inv_l, acc[7] * inv_l));
  if (r == 0 && ch == 0 && p.lse != nullptr)
    p.lse[qrow] = lsum > 0.f ? (mx + log2f(lsum)) * 0.69314718055994530942f : -INFINITY;
}

// The cluster's tokens in order.  Before the epilogue of token m the warps load
// Q of token m + 1 (once QFree says the score MMAs of token m are complete),
// so the next token's first score tiles are computed while O of token m is
// read out; after reading O they arrive on OFree.
template <bool kInt8, int kMode>
__device__ void softmax_role(const Params& p, const Ctx& c, int warp, int lane) {
  const int q = warp & 3;          // TMEM lane quadrant
  const int half = warp >> 2;      // key columns [32 half, 32 half + 32)
  const int h = q * 32 + lane;     // head
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tR = c.tmem + lane_off + kTmemRegion;  // + 64 * (i % kRegions)
  const uint32_t tO = c.tmem + lane_off + kTmemO + 128 * half;
  const bool live = h < p.n_q;
  if constexpr (kInt8)
    load_q_softmax(p, c, h, half, live, static_cast<int64_t>(token_of<kMode>(p, c, 0)) * p.n_q + h,
                   c.tmem + lane_off + kTmemQ);
  const uint32_t peer = c.crank ^ 1u;
  const uint32_t dep_zero = *reinterpret_cast<volatile uint32_t*>(c.smem + kOffZero);
  float* pair = reinterpret_cast<float*>(c.smem + kOffPair);
  const uint64_t* vmask = reinterpret_cast<const uint64_t*>(c.smem + kOffVmask);
  const float scl = p.scale_log2;
  // scores enter exp2 as fma(s, mul, -m): the raw score times the scale for a
  // positive scale (so the row max can be taken on raw scores), otherwise the
  // score is scaled first and mul = 1
  const bool raw_max = scl > 0.f;
  const float mul = raw_max ? scl : 1.f;
  int pa = 0;    // uses of the row-max / row-sum pair barrier so far (its phase)
  for (int mt = 0; mt < c.ntok; ++mt) {
    const int64_t qrow = static_cast<int64_t>(token_of<kMode>(p, c, mt)) * p.n_q + h;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int jb = seg_begin<kMode>(p, c, mt), je = seg_end<kMode>(p, c, mt);
    for (int j = jb; j < je; ++j) {  // positions in the cluster's tile stream
      {
        // own partial score tile i, read out at once so the next score MMA can
        // start while the peer's partial is still on its way
        const uint32_t reg = tR + 64 * (j % kRegions);
        if (!warp_wait(c, kBarSFull + j % kRegions, (j / kRegions) & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t own[32];
        tmem_ld_32x32b_x32(reg + 32 * half, own);
        tmem_wait_ld();
        tc_fence_before();  // ordered before the row-max handshake that precedes P(i) stores
        // the peer's partial for this warp's key columns (column half `half`)
        if (!warp_wait_cluster(c, kBarRecvFull + half, j & 1)) { ok = false; break; }
        // arm this half's next phase before the buffer is freed (the peer copies
        // into it only after that), so each phase is armed exactly once
        if (lane == 0 && q == 0 && j + 1 < c.total) mbar_arrive_expect_tx(c.bar(kBarRecvFull + half), kXchgBytes);
        float s[32];
        const uint32_t slot = c.sbase + kOffRecv + half * kXchgBytes;
        uint32_t dep = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 v = lds16f(slot + xchg_offset(h, k));
          s[4 * k + 0] = __uint_as_float(own[4 * k + 0]) + v.x;
          s[4 * k + 1] = __uint_as_float(own[4 * k + 1]) + v.y;
          s[4 * k + 2] = __uint_as_float(own[4 * k + 2]) + v.z;
          s[4 * k + 3] = __uint_as_float(own[4 * k + 3]) + v.w;
          dep ^= __float_as_uint(v.x) ^ __float_as_uint(v.w);
        }
        // Free the slot for the peer.  The arrive's address depends on every
        // loaded value (dep & dep_zero, a run-time 0), so it cannot issue
        // before the loads have returned and needs no release fence.
        mbar_arrive_remote_relaxed(mapa_shared(c.bar(kBarPeerFree + half), peer) + (dep & dep_zero));
        // mask (waiting on the stage barrier acquires the gather's validity bits) and scale
        if (!warp_wait(c, kBarFull + (j % kStages), (j / kStages) & 1)) { ok = false; break; }
        const uint32_t vm = static_cast<uint32_t>(vmask[j % kStages] >> (32 * half));
        if (!raw_max) {
#pragma unroll
          for (int k = 0; k < 32; ++k) s[k] *= scl;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          s[k] = ((vm >> k) & 1u) ? s[k] : -INFINITY;
          mx = fmaxf(mx, s[k]);
        }
        // Row max across the two column halves of head h: post, wait until both
        // posted, read.  Use pa of the pair barrier (one per tile, one per
        // token's row sum) takes slot pa % 2, so a slot is rewritten only two
        // uses later, after the partner has passed the next handshake (and so
        // has read it).
        float* slot_p = pair + (pa & 1) * 2 * kHeads;
        slot_p[half * kHeads + h] = mx;
        mbar_arrive(c.bar(kBarPairA + q));
        if (!warp_wait(c, kBarPairA + q, pa & 1)) { ok = false; break; }
        ++pa;
        mx = fmaxf(mx, slot_p[(half ^ 1) * kHeads + h]) * mul;  // log2-scaled row max of the tile
        // Lazy rescale: m only moves when the tile max exceeds it by more than 8
        // (log2 units), so P stays below 2^8 and O is rescaled rarely.
        const bool grow = mx > m + 8.f;
        const float f = grow ? fast_exp2(m - mx) : 1.f;  // m = -inf -> 0
        if (grow) {
          l *= f;
          m = mx;
        }
        if (__any_sync(0xffffffffu, grow) && j > jb) {
          // O may only be rescaled once P(j-1).V has been accumulated into it
          if (!warp_wait(c, kBarPvDone + (j - 1) % kRegions, ((j - 1) / kRegions) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + 32 * ch, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            tmem_st_32x32b_x32(tO + 32 * ch, o);
          }
          tmem_wait_st();
        }
        const float mm = (m == -INFINITY) ? 0.f : m;
        uint32_t phi[16], plo[16];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = fast_exp2(fmaf(s[2 * k], mul, -mm));
          const float p1 = fast_exp2(fmaf(s[2 * k + 1], mul, -mm));
          lsum += p0 + p1;
          const uint32_t hw = pack_bf16x2(p0, p1);
          phi[k] = hw;
          // p - bf16(p) is exact in fp32; its bf16 rounding leaves an error <= 2^-18 p
          plo[k] = pack_bf16x2(p0 - __uint_as_float(hw << 16), p1 - __uint_as_float(hw & 0xFFFF0000u));
        }
        l += lsum;
        // P(i) overwrites S(i) in its region: the senders must have read it out
        // (this warp and its pair partner read their own columns before the
        // row-max handshake above)
        if (!warp_wait(c, kBarSFree + j % kRegions, (j / kRegions) & 1)) { ok = false; break; }
        tc_fence_after();
        tmem_st_32x32b_x16(reg + 16 * half, phi);
        tmem_st_32x32b_x16(reg + 32 + 16 * half, plo);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(c.bar(kBarPFull + j % kRegions));
      }

    }
    if (!ok) return;
    if constexpr (kInt8) {
      if (mt + 1 < c.ntok) {
        // the next token's Q replaces this one's once its score MMAs are complete
        if (!warp_wait(c, kBarQFree, mt & 1)) return;
        tc_fence_after();
        load_q_softmax(p, c, h, half, live, static_cast<int64_t>(token_of<kMode>(p, c, mt + 1)) * p.n_q + h,
                       c.tmem + lane_off + kTmemQ);
      }
    }
    // l over the whole row: add the partner's column half (same order in both threads)
    float* slot_l = pair + (pa & 1) * 2 * kHeads;
    slot_l[half * kHeads + h] = l;
    mbar_arrive(c.bar(kBarPairA + q));
    if (!warp_wait(c, kBarPairA + q, pa & 1)) return;
    ++pa;
    const float l_tot = half == 0 ? l + slot_l[kHeads + h] : slot_l[h] + l;
    const int jl = je - 1;  // the segment's last tile
    if (!warp_wait(c, kBarPvDone + jl % kRegions, (jl / kRegions) & 1)) return;
    tc_fence_after();
    if constexpr (kMode == kModeListsCut) {
      if (je - jb < p.n_tiles) {
        // the token's tiles are cut between clusters: store this part's state
        store_part(p, c, token_of<kMode>(p, c, mt), h, half, live, tO, m, l_tot);
        continue;
      }
    }
    const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;
    uint4* op = reinterpret_cast<uint4*>(p.out + qrow * 512 + c.crank * 256 + half * 128);
#pragma unroll 1
    for (int ch = 0; ch < 4; ch += 2) {
      uint32_t o[64];  // two 32-column chunks per TMEM wait
      tmem_ld_32x32b_x32(tO + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(o));
      tmem_ld_32x32b_x32(tO + 32 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
      tmem_wait_ld();
      uint4 w[8];  // this head's 128-byte line of out: dims [32 ch, 32 ch + 64) of the CTA's column half
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        w[k].x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
        w[k].y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
        w[k].z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
        w[k].w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
      }
      if (p.out32) {
        // A warp's 32 heads lie 1 KB apart in out.  Each group of four lanes
        // transposes its four lines (2 butterfly stages over 32-byte pieces),
        // after which lane l of the group holds piece l of the group's e-th
        // head; the group then writes each head's 128-byte line whole.
        transpose4x32(w, lane);
        const int l4 = lane & 3;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dl = (lane & ~3) + e;  // lane of the head written
          if (q * 32 + dl < p.n_q)
            stg32(op + static_cast<int64_t>(dl - lane) * 64 + ch * 4 + 2 * l4, w[2 * e], w[2 * e + 1]);
        }
      } else if (live) {
#pragma unroll
        for (int k = 0; k < 8; ++k) op[ch * 4 + k] = w[k];
      }
    }
    // O is in registers: the next token's first P.V may overwrite it
    tc_fence_before();
    mbar_arrive(c.bar(kBarOFree));
    if (live && c.crank == 0 && half == 0 && p.lse != nullptr)
      p.lse[qrow] = l_tot > 0.f ? (m + log2f(l_tot)) * 0.69314718055994530942f : -INFINITY;
  }
}

// ------------------------------------------------------------------ kernel
// kMode: top-k lists, a sliding window, or a window plus compressed-cache
// entries (separate instantiations, so each compiles only its own path).
template <bool kInt8, int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) mla_sparse_fwd_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Ctx c;
  c.smem = smem;
  c.sbase = smem_u32(smem);
  c.crank = cluster_ctarank();
  c.cid = blockIdx.x >> 1;
  if constexpr (kMode == kModeListsCut) {
    c.first = cluster_start(p, c.cid);
    c.total = cluster_start(p, c.cid + 1) - c.first;
    c.tok0 = c.first / p.n_tiles;
    c.ntok = (c.first + c.total - 1) / p.n_tiles - c.tok0 + 1;
  } else {
    c.first = 0;
    c.tok0 = c.cid;
    c.ntok = (p.T - c.cid + p.n_clusters - 1) / p.n_clusters;
    c.total = c.ntok * p.n_tiles;
  }
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
  c.wait_ns = p.wait_ns;
  if (tid == 0) {
    // the swizzled operand layouts need a 1024-byte aligned base
    const bool misaligned = (c.sbase & 1023u) != 0;
    *c.abort = misaligned ? 1u : 0u;
    if (misaligned) atomicOr(&g_mla_status, MLA_DEVICE_TIMEOUT);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(c.bar(kBarFull + i), kInt8 ? 256 : 256 + 8);
      mbar_init(c.bar(kBarEmpty + i), 1);
    }
    for (int i = 0; i < kIdxSlots; ++i) {
      mbar_init(c.bar(kBarIdxFull + i), 32);
      mbar_init(c.bar(kBarIdxEmpty + i), 256);
    }
    for (int r = 0; r < kRegions; ++r) {
      mbar_init(c.bar(kBarSFull + r), 1);
      mbar_init(c.bar(kBarSFree + r), kSenderThreads);
      mbar_init(c.bar(kBarPFull + r), kSoftmaxThreads);
      mbar_init(c.bar(kBarPvDone + r), 1);
    }
    for (int h2 = 0; h2 < 2; ++h2) {
      mbar_init(c.bar(kBarRecvFull + h2), 1);
      mbar_init(c.bar(kBarPeerFree + h2), kSoftmaxThreads / 2);  // the four warps reading that column half
    }
    for (int q = 0; q < 4; ++q) mbar_init(c.bar(kBarPairA + q), 64);
    mbar_init(c.bar(kBarQReady), kInt8 ? kSoftmaxThreads : kSenderThreads);
    mbar_init(c.bar(kBarQFree), 1);
    mbar_init(c.bar(kBarOFree), kSoftmaxThreads);
    mbar_init(c.bar(kBarFinal), 1);
    fence_mbarrier_init_cluster();
    for (int h2 = 0; h2 < 2; ++h2) mbar_arrive_expect_tx(c.bar(kBarRecvFull + h2), kXchgBytes);
    *reinterpret_cast<volatile uint32_t*>(smem + kOffZero) = 0u;
    *reinterpret_cast<volatile int*>(smem + kOffTotal) = c.total;
  }
  // the index warps issue their first top-k loads before the set-up barrier
  int idx0[8];
  if (warp >= kIndexWarp && warp < kIndexWarp + kIndexWarps)
    index_load<kMode>(p, c, (warp - kIndexWarp) * kIdxBatch, lane, idx0);
  if (warp == kMmaWarp) {
    tmem_alloc(c.sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  c.tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp < kSenderWarp0) {
    regs_increase<Regs<kInt8>::kSoftmax>();
    if (!*c.abort) softmax_role<kInt8, kMode>(p, c, warp, lane);
  } else if (warp < kGatherWarp0) {
    if (!*c.abort) sender_role<kInt8, kMode>(p, c, warp - kSenderWarp0, lane);
  } else if (warp < kMmaWarp) {
    regs_decrease<Regs<kInt8>::kGather>();
    if (!*c.abort) gather_role<kInt8, kMode>(p, c, warp - kGatherWarp0, lane);
  } else {
    regs_decrease<Regs<kInt8>::kControl>();
    if (!*c.abort) {
      if (warp == kMmaWarp) {
        if (lane == 0) mma_role<kMode>(p, c);
        __syncwarp();
      } else if (warp < kIndexWarp + kIndexWarps) {
        index_role<kMode>(p, c, warp - kIndexWarp, lane, idx0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(c.tmem, kTmemCols);
  if (tid == 0 && *c.abort) atomicOr(&g_mla_status, MLA_DEVICE_TIMEOUT);
  // Neither CTA may exit while its peer could still address its shared memory.
  cluster_arrive();
  cluster_wait();
}

}  // namespace mlasp

// ==================================================================== C ABI
namespace {

thread_local char g_last_error[512] = "";

mla_status fail(mla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mla_status fail(mla_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

constexpr int kMaxDevices = 64;
// kernel variants: kv = int8 + 2 * mode (mode kModeLists .. kModeListsCut)
constexpr int kVariants = 8;
std::once_flag g_attr_once[kMaxDevices][kVariants];
cudaError_t g_attr_err[kMaxDevices][kVariants];

int g_max_clusters[kMaxDevices][kVariants];

// Per (device, stream) buffer for the partial softmax states of cut tokens:
// one slot per (cluster, first/last token, CTA rank).  Allocated by the first
// call on a stream that cuts tokens (not under graph capture) and kept for the
// life of the process.
struct CutBuffer {
  int dev;
  void* stream;
  float* ws;
  int clusters;
};
std::mutex g_cut_mu;
CutBuffer* g_cut = nullptr;
int g_cut_n = 0, g_cut_cap = 0;

// The buffer for (dev, stream), or nullptr when there is none and none may be
// made now (the stream is capturing a graph) or the allocation failed (*err).
float* cut_buffer(int dev, cudaStream_t stream, int clusters, cudaError_t* err) {
  std::lock_guard<std::mutex> lock(g_cut_mu);
  *err = cudaSuccess;
  for (int i = 0; i < g_cut_n; ++i) {
    const CutBuffer& b = g_cut[i];
    if (b.dev == dev && b.stream == static_cast<void*>(stream) && b.clusters >= clusters) return b.ws;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
  if (g_cut_n == g_cut_cap) {
    const int cap = g_cut_cap ? 2 * g_cut_cap : 8;
    CutBuffer* nb = static_cast<CutBuffer*>(realloc(g_cut, sizeof(CutBuffer) * cap));
    if (nb == nullptr) return nullptr;
    g_cut = nb;
    g_cut_cap = cap;
  }
  void* mem = nullptr;
  const cudaError_t e = cudaMalloc(&mem, static_cast<size_t>(clusters) * 4 * mlasp::kSlotFloats * sizeof(float));
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  CutBuffer& b = g_cut[g_cut_n++];
  b.dev = dev;
  b.stream = static_cast<void*>(stream);
  b.ws = static_cast<float*>(mem);
  b.clusters = clusters;
  return b.ws;
}

// Equal shares give each cluster at least this many tiles.
constexpr int64_t kMinPartTiles = 2;

// Kernel launches enqueued by the attention entry points.
std::atomic<unsigned long long> g_launches{0};
// Whether calls may cut tokens between clusters (and so allocate the buffer).
std::atomic<int> g_allow_cut{1};

// Bound of every device-side wait of the next launches (nanoseconds).
std::atomic<unsigned long long> g_wait_ns{500ull * 1000ull * 1000ull};

// Also records how many two-CTA clusters of the kernel the device runs at once.
template <bool kInt8, int kMode>
cudaError_t prepare_kernel(int dev) {
  constexpr int kv = (kInt8 ? 1 : 0) + 2 * kMode;
  std::call_once(g_attr_once[dev][kv], [dev] {
    cudaError_t e = cudaFuncSetAttribute(mlasp::mla_sparse_fwd_kernel<kInt8, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, mlasp::kSmemBytes);
    if (e == cudaSuccess) {
      // The warpgroups re-divide the registers the block is launched with;
      // refuse to launch if the compiled per-thread count cannot cover them.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, mlasp::mla_sparse_fwd_kernel<kInt8, kMode>);
      using R = mlasp::Regs<kInt8>;
      const long need = 256L * R::kSoftmax + 128L * 80 + 256L * R::kGather + 128L * R::kControl;
      if (e == cudaSuccess && (fa.numRegs < 80 || static_cast<long>(fa.numRegs) * mlasp::kThreads < need))
        e = cudaErrorInvalidConfiguration;
    }
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(mlasp::kThreads, 1, 1);
      cfg.dynamicSmemBytes = mlasp::kSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, mlasp::mla_sparse_fwd_kernel<kInt8, kMode>, &cfg);
      g_max_clusters[dev][kv] = n;
      if (e == cudaSuccess && n < 1) e = cudaErrorInvalidConfiguration;
    }
    g_attr_err[dev][kv] = e;
  });
  return g_attr_err[dev][kv];
}

}  // namespace

namespace mlasp {
// The bound of every device-side wait, read by each of the library's launches.
unsigned long long host_wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace mlasp

extern "C" {

int32_t mla_sparse_abi_version(void) { return 202; }

const char* mla_sparse_last_error(void) { return g_last_error; }

}  // extern "C"

namespace {

// Shared by the entry points: window == 0 reads the top-k lists, window > 0
// builds each token's sliding window, followed by compressed-cache entries when
// `cmp` is given (d.topk is then the number of entries per token).
mla_status attn_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope, const void* kv_nope,
                    const void* kv_rope, const float* kv_scales, const int32_t* topk_idx, int32_t window,
                    const mla_cmp_cache* cmp, const int32_t* block_table, const int32_t* act_seqs, void* out,
                    float* lse, float softmax_scale, int32_t mode, void* stream) {
  g_last_error[0] = '\0';
  if (dims == nullptr) return fail(MLA_ERR_NULL, "dims is NULL");
  mla_dims d = *dims;
  if (window < 0) return fail(MLA_ERR_SHAPE, "window=%d must be >= 1", window);
  int cmp_slots = 0;
  if (cmp != nullptr) {
    if (!cmp->nope || !cmp->rope || !cmp->block_table || (d.kv_dtype == MLA_KV_INT8 && !cmp->scales))
      return fail(MLA_ERR_NULL, "a required compressed-cache pointer is NULL");
    if (cmp->ratio < 1 || cmp->num_blocks < 1 || cmp->max_blocks_per_seq < 1 || (cmp->sparse_idx && cmp->topk < 1))
      return fail(MLA_ERR_SHAPE, "compressed cache: ratio, num_blocks, max_blocks_per_seq (and topk for SCFA) must be >= 1");
    if (cmp->num_blocks >= (1 << 23) || d.num_blocks >= (1 << 23))
      return fail(MLA_ERR_SHAPE, "with a compressed cache both caches need num_blocks < 2^23");
    if (!aligned(cmp->nope, 16) || !aligned(cmp->rope, 16) || (cmp->scales && !aligned(cmp->scales, 16)) ||
        !aligned(cmp->block_table, 4) || (cmp->sparse_idx && !aligned(cmp->sparse_idx, 4)))
      return fail(MLA_ERR_ALIGN, "compressed-cache rows must be 16-byte, tables 4-byte aligned");
    // CFA: as many slots as the longest sequence can have compressed entries
    const int64_t most = std::min<int64_t>(static_cast<int64_t>(cmp->max_blocks_per_seq) * 128,
                                           static_cast<int64_t>(d.max_blocks_per_seq) * 128 / cmp->ratio);
    cmp_slots = cmp->sparse_idx ? cmp->topk : static_cast<int>(most);
  }
  if (window > 0) {
    if (static_cast<int64_t>(window) + cmp_slots > (1 << 24))
      return fail(MLA_ERR_SHAPE, "window + compressed entries per token too large");
    d.topk = window + cmp_slots;
  }
  if (!q_nope || !q_rope || !kv_nope || !kv_rope || (window == 0 && !topk_idx) || !block_table || !act_seqs || !out)
    return fail(MLA_ERR_NULL, "a required tensor pointer is NULL");
  if (d.kv_dtype != MLA_KV_BF16 && d.kv_dtype != MLA_KV_INT8)
    return fail(MLA_ERR_DTYPE, "kv_dtype %d is neither MLA_KV_BF16 nor MLA_KV_INT8", d.kv_dtype);
  if (d.kv_dtype == MLA_KV_INT8 && kv_scales == nullptr)
    return fail(MLA_ERR_DTYPE, "kv_scales is required for an INT8 cache");
  if (d.B < 1 || d.S1 < 1 || d.topk < 1 || d.num_blocks < 1 || d.max_blocks_per_seq < 1)
    return fail(MLA_ERR_SHAPE, "B, S1, topk, num_blocks and max_blocks_per_seq must be >= 1");
  if (d.n_q < 1 || d.n_q > 128) return fail(MLA_ERR_SHAPE, "n_q=%d outside [1, 128]", d.n_q);
  if (d.n_kv != 1) return fail(MLA_ERR_UNSUPPORTED, "n_kv=%d: only one latent KV head is implemented", d.n_kv);
  if (d.d_nope != 512 || d.d_rope != 64 || d.block_size != 128)
    return fail(MLA_ERR_UNSUPPORTED, "d_nope=%d d_rope=%d block_size=%d: only 512/64/128 are implemented", d.d_nope,
                d.d_rope, d.block_size);
  if (d.num_blocks >= (1 << 24)) return fail(MLA_ERR_SHAPE, "num_blocks=%d must be < 2^24", d.num_blocks);
  const int64_t T = static_cast<int64_t>(d.B) * d.S1;
  if (T > (1ll << 30)) return fail(MLA_ERR_SHAPE, "B*S1=%lld too large", static_cast<long long>(T));
  if (mode != MLA_MODE_DECODE && mode != MLA_MODE_PREFILL) return fail(MLA_ERR_SHAPE, "mode %d unknown", mode);
  if (!isfinite(softmax_scale)) return fail(MLA_ERR_SHAPE, "softmax_scale is not finite");
  if (!aligned(q_nope, 16) || !aligned(q_rope, 16) || !aligned(kv_nope, 16) || !aligned(kv_rope, 16) ||
      !aligned(out, 16) || (kv_scales && d.kv_dtype == MLA_KV_INT8 && !aligned(kv_scales, 16)))
    return fail(MLA_ERR_ALIGN, "q/kv/out/scales pointers must be 16-byte aligned");
  if ((topk_idx && !aligned(topk_idx, 4)) || !aligned(block_table, 4) || !aligned(act_seqs, 4) || (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_ALIGN, "index tensors and lse must be 4-byte aligned");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
  const bool int8 = d.kv_dtype == MLA_KV_INT8;
  const int kmode = cmp != nullptr ? mlasp::kModeCompressed : (window > 0 ? mlasp::kModeWindow : mlasp::kModeLists);
  int kv = (int8 ? 1 : 0) + 2 * kmode;
  switch (kv) {
    case 0: e = prepare_kernel<false, mlasp::kModeLists>(dev); break;
    case 1: e = prepare_kernel<true, mlasp::kModeLists>(dev); break;
    case 2: e = prepare_kernel<false, mlasp::kModeWindow>(dev); break;
    case 3: e = prepare_kernel<true, mlasp::kModeWindow>(dev); break;
    case 4: e = prepare_kernel<false, mlasp::kModeCompressed>(dev); break;
    default: e = prepare_kernel<true, mlasp::kModeCompressed>(dev); break;
  }
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "kernel set-up: %s", cudaGetErrorString(e));

  mlasp::Params p;
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.kv_nope = kv_nope;
  p.kv_rope = static_cast<const uint16_t*>(kv_rope);
  p.kv_scales = int8 ? kv_scales : nullptr;
  p.topk_idx = topk_idx;
  p.block_table = block_table;
  p.act_seqs = act_seqs;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.S1 = d.S1;
  p.n_q = d.n_q;
  p.topk = d.topk;
  p.num_blocks = d.num_blocks;
  p.mbps = d.max_blocks_per_seq;
  p.n_tiles = (d.topk + mlasp::kTileKeys - 1) / mlasp::kTileKeys;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
  p.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  // Persistent clusters, as many as run at once.  Whole tokens per cluster by
  // default.  Equal shares of tiles (list mode only) cost a token switch per
  // cut, a merge launch and the L2 sharing between a sequence's tokens; they
  // are taken when whole tokens would leave the longest cluster at least
  // twice the equal share (few tokens with long lists, most clusters idle).
  const int max_clusters = g_max_clusters[dev][kv];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.T = static_cast<int>(T);
  const int64_t tiles = T * p.n_tiles;
  if (tiles >= (1ll << 31) - p.n_tiles)
    return fail(MLA_ERR_SHAPE, "B*S1 x key tiles per token = %lld too large", static_cast<long long>(tiles));
  p.ws = nullptr;
  p.n_clusters = static_cast<int>(T < max_clusters ? T : max_clusters);
  if (kmode == mlasp::kModeLists && g_allow_cut.load(std::memory_order_relaxed)) {
    const int64_t nc_equal = std::min<int64_t>(max_clusters, std::max<int64_t>(1, tiles / kMinPartTiles));
    const int64_t most_whole = (T + p.n_clusters - 1) / p.n_clusters * p.n_tiles;
    const int64_t most_equal = (tiles + nc_equal - 1) / nc_equal;
    if (most_whole >= 2 * most_equal && most_whole >= 4) {
      p.ws = cut_buffer(dev, s, max_clusters, &e);
      if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "buffer for cut tokens: %s", cudaGetErrorString(e));
      if (p.ws != nullptr) {
        e = int8 ? prepare_kernel<true, mlasp::kModeListsCut>(dev) : prepare_kernel<false, mlasp::kModeListsCut>(dev);
        if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "kernel set-up: %s", cudaGetErrorString(e));
        kv = (int8 ? 1 : 0) + 2 * mlasp::kModeListsCut;
        p.n_clusters = static_cast<int>(std::min<int64_t>(nc_equal, g_max_clusters[dev][kv]));
      }
    }
  }
  p.window = window;
  p.cmp_nope = cmp ? cmp->nope : nullptr;
  p.cmp_rope = cmp ? static_cast<const uint16_t*>(cmp->rope) : nullptr;
  p.cmp_scales = cmp && int8 ? cmp->scales : nullptr;
  p.cmp_block_table = cmp ? cmp->block_table : nullptr;
  p.cmp_idx = cmp ? cmp->sparse_idx : nullptr;
  p.cmp_num_blocks = cmp ? cmp->num_blocks : 0;
  p.cmp_mbps = cmp ? cmp->max_blocks_per_seq : 0;
  p.cmp_ratio = cmp ? cmp->ratio : 1;
  p.cmp_topk = cmp_slots;
  const dim3 grid(static_cast<unsigned>(2 * p.n_clusters));
  switch (kv) {
    case 0: mlasp::mla_sparse_fwd_kernel<false, mlasp::kModeLists><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 1: mlasp::mla_sparse_fwd_kernel<true, mlasp::kModeLists><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 2: mlasp::mla_sparse_fwd_kernel<false, mlasp::kModeWindow><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 3: mlasp::mla_sparse_fwd_kernel<true, mlasp::kModeWindow><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 4: mlasp::mla_sparse_fwd_kernel<false, mlasp::kModeCompressed><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 5: mlasp::mla_sparse_fwd_kernel<true, mlasp::kModeCompressed><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    case 6: mlasp::mla_sparse_fwd_kernel<false, mlasp::kModeListsCut><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
    default: mlasp::mla_sparse_fwd_kernel<true, mlasp::kModeListsCut><<<grid, mlasp::kThreads, mlasp::kSmemBytes, s>>>(p); break;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (p.ws != nullptr) {
    // merge the cut tokens' parts; launched early, it waits for the kernel above
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(T), 2, 256 / mlasp::kCombineDims);
    cfg.blockDim = dim3(mlasp::kHeads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mlasp::combine_kernel, p);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status mla_sparse_attn_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope, const void* kv_nope,
                               const void* kv_rope, const float* kv_scales, const int32_t* topk_idx,
                               const int32_t* block_table, const int32_t* act_seqs, void* out, float* lse,
                               float softmax_scale, int32_t mode, void* stream) {
  return attn_fwd(dims, q_nope, q_rope, kv_nope, kv_rope, kv_scales, topk_idx, 0, nullptr, block_table, act_seqs, out,
                  lse, softmax_scale, mode, stream);
}

mla_status mla_swa_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope, const void* kv_nope,
                       const void* kv_rope, const float* kv_scales, const int32_t* block_table,
                       const int32_t* act_seqs, int32_t window, void* out, float* lse, float softmax_scale,
                       int32_t mode, void* stream) {
  if (window < 1) {
    g_last_error[0] = '\0';
    return fail(MLA_ERR_SHAPE, "window=%d must be >= 1", window);
  }
  return attn_fwd(dims, q_nope, q_rope, kv_nope, kv_rope, kv_scales, nullptr, window, nullptr, block_table, act_seqs,
                  out, lse, softmax_scale, mode, stream);
}

mla_status mla_compressed_attn_fwd(const mla_dims* dims, const void* q_nope, const void* q_rope, const void* kv_nope,
                                   const void* kv_rope, const float* kv_scales, const int32_t* block_table,
                                   const mla_cmp_cache* cmp, const int32_t* act_seqs, int32_t window, void* out,
                                   float* lse, float softmax_scale, int32_t mode, void* stream) {
  if (window < 1 || cmp == nullptr) {
    g_last_error[0] = '\0';
    return fail(window < 1 ? MLA_ERR_SHAPE : MLA_ERR_NULL, window < 1 ? "window=%d must be >= 1" : "cmp is NULL (window %d)",
                window);
  }
  return attn_fwd(dims, q_nope, q_rope, kv_nope, kv_rope, kv_scales, nullptr, window, cmp, block_table, act_seqs, out,
                  lse, softmax_scale, mode, stream);
}

mla_status mla_sparse_set_wait_limit_ns(uint64_t ns) {
  g_last_error[0] = '\0';
  if (ns < 1000ull || ns > 60ull * 1000ull * 1000ull * 1000ull)
    return fail(MLA_ERR_SHAPE, "wait limit %llu ns outside [1 us, 60 s]", static_cast<unsigned long long>(ns));
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return MLA_OK;
}

mla_status mla_sparse_get_device_status(void* stream) { return mla_sparse_device_status(stream, nullptr, 0); }

uint64_t mla_sparse_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void mla_sparse_allow_cut_tokens(int32_t allow) { g_allow_cut.store(allow ? 1 : 0, std::memory_order_relaxed); }

mla_status mla_sparse_device_status(void* stream, uint32_t* flags, int32_t clear) {
  g_last_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, mlasp::g_mla_status, sizeof v);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(mlasp::g_mla_status, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  if (flags) *flags = v;
  if (v != 0) return fail(MLA_ERR_DEVICE_STATUS, "device status 0x%x", v);
  return MLA_OK;
}

}  // extern "C"
