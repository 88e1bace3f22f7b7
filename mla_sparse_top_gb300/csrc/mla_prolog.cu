// MLA Prolog for GB300 (sm_103a): hidden states to the absorbed query of the
// sparse attention, plus the new key row written into its paged cache.
//
// Formulas: "NPU DeepSeek-V4 PyPTO fused-operator optimization", section
// MlaProlog (query: two projections, each followed by an RMSNorm, the second
// with weight 1, interleaved RoPE on the last rope_dim; key: one projection,
// RMSNorm, RoPE on the last rope_dim); "CANN DeepSeek Indexer attention",
// section MLA Prolog (weight absorption in decode: the query's no-position
// part is taken into the 512-wide latent space by w_uk).
//
// Data flow per call (T tokens, H heads), five launches on the caller's stream:
//   gemm_kernel   c_raw = x @ wq_a and kv_raw = x @ wkv in one launch (the
//                 page runs the two projections side by side), fp32 partial
//                 sums over k splits in separate slots
//   x_rows_kernel one block per token: c^Q = bf16(RMSNorm(sum of c_raw
//                 slots) * gamma_cq) by four warps; k = RMSNorm(sum of
//                 kv_raw slots) * gamma_ckv, RoPE on k[512:], rounded to bf16
//                 and written (bf16 or INT8) into the cache row by the fifth
//   gemm_kernel   q_raw = c^Q @ wq_b, fp32 slots
//   q_heads_kernel  per (t, h) RMSNorm over 192 of the summed slots, q[:128]
//                 -> bf16 operand, RoPE(q[128:]) -> q_rope
//   gemm_kernel   q_nope[h] = q[h][:128] @ w_uk[h] for every head, bf16 out
// The matrix products are this file's tcgen05 kernel: the weights stream
// through a TMA ring as the MMA's A operand (M = 128 output features,
// MN-major: the weights' own row-major layout), the tokens are N (up to 256
// per work unit), the accumulators double-buffer in TMEM so one unit's
// epilogue overlaps the next unit's loads.  The norms are memory-bound row
// passes in fp32 with one rounding to bf16 at each storage point: four warps
// per c^Q row, a warp per key row and per (token, head);
// they sum the k-split slots in a fixed order, so the result does not depend
// on scheduling.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <utility>

#include "../../include/mla_prolog.h"
#include "ptx.cuh"

namespace mlasp {
unsigned long long host_wait_limit_ns();  // the library's wait bound (mla_sparse_set_wait_limit_ns)
}

namespace mlapro {
using namespace mlasp;

constexpr int kWarps = 8;
constexpr int kQkNope = 128;
constexpr int kRope = 64;
constexpr int kLatent = 512;
constexpr int kKv = kLatent + kRope;  // 576
constexpr int kQHead = kQkNope + kRope;  // 192

__device__ unsigned int g_prolog_status = 0;

struct NormParams {
  const float* c_raw;        // [c_slots][T, q_lora] partial sums
  const uint16_t* gamma_cq;  // bf16 [q_lora]
  uint16_t* c_q;             // bf16 [T, q_lora]
  const float* kv_raw;       // [kv_slots][T, 576] partial sums
  const uint16_t* gamma_ckv; // bf16 [576]
  const float* cos;          // [T, 32]
  const float* sin;
  const int64_t* idx;        // [T]
  uint8_t* kv_nope;
  uint8_t* kv_rope;
  float* kv_scales;
  int64_t num_rows;
  int q_lora;
  int T;
  int int8;
  int c_slots, kv_slots;
  float eps;
};

struct HeadParams {
  const float* q_raw;  // [q_slots][T * H, 192] partial sums
  const float* cos;
  const float* sin;
  uint16_t* q_n;       // bf16 [T * H, 128]
  uint16_t* q_rope;    // bf16 [T * H, 64]
  int H;
  int TH;
  int q_slots;
  float eps;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values rounded (nearest, ties to even) into one bf16 pair, low half first.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 1 / sqrt(mean + eps), the reciprocal square root correctly rounded.
__device__ __forceinline__ float inv_rms(float sumsq, int n, float eps) {
  return __frsqrt_rn(__fadd_rn(__fdiv_rn(sumsq, static_cast<float>(n)), eps));
}

// The INT8 rule of the cache: code = clamp(round half to even (x / scale)) with the division in fp32.
__device__ __forceinline__ uint32_t code8(float x, float scale) {
  const int q = __float2int_rn(__fdiv_rn(x, scale));
  return static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(max(-128, min(127, q)))));
}

constexpr int kCqThreads = 128;  // warps 0-3 of a row block: the c^Q row
constexpr int kRowThreads = kCqThreads + 32;  // warp 4: the key row
constexpr int kStageCqMax = 12288;  // c^Q rows up to this width are summed once into shared memory

// The c^Q row of token t by threads 0..127: sum of squares over the row (the
// slots summed in slot order, staged in shared memory when `stage` is given),
// then the scaled, rounded row.
__device__ __forceinline__ void cq_row(const NormParams& p, int t, int tid, float* stage) {
  __shared__ float part[kCqThreads / 32];
  const float4* src = reinterpret_cast<const float4*>(p.c_raw + static_cast<int64_t>(t) * p.q_lora);
  const int64_t slot4 = static_cast<int64_t>(p.T) * p.q_lora / 4;  // one k-split slot, in float4
  const int n4 = p.q_lora >> 2;
  auto row4 = [&](int i) {  // the slots summed in slot order
    float4 v = src[i];
#pragma unroll 4
    for (int k = 1; k < p.c_slots; ++k) {
      const float4 w = src[k * slot4 + i];
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    return v;
  };
  float4* st4 = reinterpret_cast<float4*>(stage);
  float ss = 0.f;
  for (int i = tid; i < n4; i += kCqThreads) {
    const float4 v = row4(i);
    if (stage != nullptr) st4[i] = v;  // read back below by this same thread
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  asm volatile("bar.sync 1, %0;" :: "n"(kCqThreads) : "memory");  // warps 0-3 only
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCqThreads / 32; ++w) tot += part[w];
  const float inv = inv_rms(tot, p.q_lora, p.eps);
  const uint2* gam = reinterpret_cast<const uint2*>(p.gamma_cq);
  uint2* dst = reinterpret_cast<uint2*>(p.c_q + static_cast<int64_t>(t) * p.q_lora);
  for (int i = tid; i < n4; i += kCqThreads) {
    const float4 v = stage != nullptr ? st4[i] : row4(i);
    const uint2 gw = __ldg(gam + i);
    dst[i] = make_uint2(pack_bf16(v.x * inv * bf16_lo(gw.x), v.y * inv * bf16_hi(gw.x)),
                        pack_bf16(v.z * inv * bf16_lo(gw.y), v.w * inv * bf16_hi(gw.y)));
  }
}

// The key row of token t by one warp: RMSNorm over the 576-wide row, RoPE on
// its tail, the cache write.
__device__ __forceinline__ void kv_row(const NormParams& p, int t, int lane) {
  // lane l: latent dims [16 l, 16 l + 16) (eight lanes per 128-element group) and rope pair l
  const float* row = p.kv_raw + static_cast<int64_t>(t) * kKv;
  const int64_t slot = static_cast<int64_t>(p.T) * kKv;  // one k-split slot
  float x[16];
  float2 rp = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int sl = 0; sl < p.kv_slots; ++sl) {  // the slots summed in slot order
    const float* r = row + sl * slot;
    const float4* s4 = reinterpret_cast<const float4*>(r + 16 * lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = s4[k];
      x[4 * k] = sl ? x[4 * k] + v.x : v.x;
      x[4 * k + 1] = sl ? x[4 * k + 1] + v.y : v.y;
      x[4 * k + 2] = sl ? x[4 * k + 2] + v.z : v.z;
      x[4 * k + 3] = sl ? x[4 * k + 3] + v.w : v.w;
    }
    const float2 w = reinterpret_cast<const float2*>(r + kLatent)[lane];
    rp.x = sl ? rp.x + w.x : w.x;
    rp.y = sl ? rp.y + w.y : w.y;
  }
  const float c = __ldg(p.cos + static_cast<int64_t>(t) * 32 + lane);
  const float s = __ldg(p.sin + static_cast<int64_t>(t) * 32 + lane);
  const int64_t r = __ldg(p.idx + t);
  float ss = rp.x * rp.x + rp.y * rp.y;
#pragma unroll
  for (int k = 0; k < 16; ++k) ss += x[k] * x[k];
  const float inv = inv_rms(warp_sum(ss), kKv, p.eps);
  const uint4* gam = reinterpret_cast<const uint4*>(p.gamma_ckv + 16 * lane);
  const uint4 g0 = __ldg(gam), g1 = __ldg(gam + 1);
  const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  uint32_t kb[8];  // the bf16 cache row
#pragma unroll
  for (int k = 0; k < 8; ++k)
    kb[k] = pack_bf16(x[2 * k] * inv * bf16_lo(gw[k]), x[2 * k + 1] * inv * bf16_hi(gw[k]));
  const uint32_t gr = __ldg(reinterpret_cast<const uint32_t*>(p.gamma_ckv + kLatent) + lane);
  const float a = rp.x * inv * bf16_lo(gr), b = rp.y * inv * bf16_hi(gr);
  const uint32_t rope = pack_bf16(a * c - b * s, a * s + b * c);
  if (r < 0) return;
  if (r >= p.num_rows) {
    if (lane == 0) atomicOr(&g_prolog_status, MLA_DEVICE_BAD_BLOCK);
    return;
  }
  reinterpret_cast<uint32_t*>(p.kv_rope + r * (kRope * 2))[lane] = rope;
  if (!p.int8) {
    uint4* dst = reinterpret_cast<uint4*>(p.kv_nope + r * (kLatent * 2)) + 2 * lane;
    dst[0] = make_uint4(kb[0], kb[1], kb[2], kb[3]);
    dst[1] = make_uint4(kb[4], kb[5], kb[6], kb[7]);
    return;
  }
  float xb[16];
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    xb[2 * k] = bf16_lo(kb[k]);
    xb[2 * k + 1] = bf16_hi(kb[k]);
    am = fmaxf(am, fmaxf(fabsf(xb[2 * k]), fabsf(xb[2 * k + 1])));
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  float scale = __fdiv_rn(am, 127.f);
  if (!(scale > 0.f)) scale = 1.f;
  uint32_t q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    q[k] = code8(xb[4 * k], scale) | (code8(xb[4 * k + 1], scale) << 8) | (code8(xb[4 * k + 2], scale) << 16) |
           (code8(xb[4 * k + 3], scale) << 24);
  reinterpret_cast<uint4*>(p.kv_nope + r * kLatent)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
  if ((lane & 7) == 0) p.kv_scales[r * 4 + (lane >> 3)] = scale;
}

// One block per token: warps 0-3 the c^Q row, warp 4 the key row.
__global__ void __launch_bounds__(kRowThreads) x_rows_kernel(const NormParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ float4 stage_c[];
  const int t = blockIdx.x;
  if (threadIdx.x < kCqThreads)
    cq_row(p, t, threadIdx.x, p.q_lora <= kStageCqMax ? reinterpret_cast<float*>(stage_c) : nullptr);
  else
    kv_row(p, t, threadIdx.x & 31);
}

// One warp per (token, head): lane l holds dims (2l, 2l+1), (64+2l, 65+2l) and rope pair l.
__global__ void __launch_bounds__(kWarps * 32) q_heads_kernel(const HeadParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kWarps + warp;
  if (g >= p.TH) return;
  const int t = g / p.H;
  const float2* row = reinterpret_cast<const float2*>(p.q_raw + static_cast<int64_t>(g) * kQHead);
  const int64_t slot2 = static_cast<int64_t>(p.TH) * kQHead / 2;  // one k-split slot, in float2
  float2 u = row[lane], v = row[32 + lane], w = row[64 + lane];
#pragma unroll 4
  for (int k = 1; k < p.q_slots; ++k) {  // the slots summed in slot order
    const float2 a = row[k * slot2 + lane], b = row[k * slot2 + 32 + lane], c2 = row[k * slot2 + 64 + lane];
    u.x += a.x;
    u.y += a.y;
    v.x += b.x;
    v.y += b.y;
    w.x += c2.x;
    w.y += c2.y;
  }
  const float c = __ldg(p.cos + static_cast<int64_t>(t) * 32 + lane);
  const float s = __ldg(p.sin + static_cast<int64_t>(t) * 32 + lane);
  const float ss = u.x * u.x + u.y * u.y + v.x * v.x + v.y * v.y + w.x * w.x + w.y * w.y;
  const float inv = inv_rms(warp_sum(ss), kQHead, p.eps);
  uint32_t* qn = reinterpret_cast<uint32_t*>(p.q_n + static_cast<int64_t>(g) * kQkNope);
  qn[lane] = pack_bf16(u.x * inv, u.y * inv);
  qn[32 + lane] = pack_bf16(v.x * inv, v.y * inv);
  const float a = w.x * inv, b = w.y * inv;
  reinterpret_cast<uint32_t*>(p.q_rope + static_cast<int64_t>(g) * kRope)[lane] = pack_bf16(a * c - b * s, a * s + b * c);
}

// ------------------------------------------------------------------ matrix products
// out[t, f] = sum_k X[t, k] W[k, f] for bf16 row-major X [T, K] and W [K, F]
// (W's k rows optionally offset per batch b, X's k columns likewise), fp32
// accumulation.  A work unit is (batch b, feature tile, k split s, token
// tile); its MMAs are D[f, t] (M = 128 features, N = 128 tokens, K = 16) with
// A = 128 features of the weight tile (MN-major: the weights' own row-major
// layout, 64 k rows per stage, 128-byte swizzle) and B = 128 tokens of the
// token tile (K-major, 64 k).  A unit covers fsub x tsub of these 128 x 128
// blocks (fsub * tsub = 2): with at most 128 tokens a unit spans 256
// features, so each weight row is read in 512-byte pieces (fewer DRAM pages
// opened per byte); otherwise 128 features and up to 256 tokens.  Many units keep every SM streaming weights (one SM alone does not reach its
// share of HBM bandwidth).  Out-of-range rows and columns read as zero from the TMA engine, so any T,
// K and F work.  Output: fp32 into slot s of [splits][T][F] (summed later in
// slot order) or, unsplit, bf16 into out[t * ld + b * F + f].
constexpr int kGemmThreads = 192;     // warps 0-3 epilogue (one TMEM lane quadrant each), 4 TMA, 5 MMA
constexpr int kBoxBytes = 64 * 128;   // one 64 x 64 box of bf16
// A stage holds 2 fsub weight boxes (8 KB each) and tsub 128-token halves
// (16 KB each): 48 KB, four stages.
constexpr int kGemmStageBytes = 6 * kBoxBytes;
constexpr int kGemmMaxStages = 4;
constexpr int kGemmRing = kGemmMaxStages * kGemmStageBytes;  // 192 KB
constexpr int kGemmOffBars = kGemmRing;
constexpr int kGemmBars = 2 * kGemmMaxStages + 4 + 1;  // full, empty, acc full [2], acc empty [2], final
constexpr int kGemmSmem = kGemmOffBars + kGemmBars * 8 + 16 + 1024;  // + slack to align the base to 1024
// Waits that only let MMAs already in flight complete before the CTA exits are
// never cut shorter than this, whatever the configured bound.
constexpr uint64_t kGemmDrainNs = 500ull * 1000ull * 1000ull;

struct GemmJob {
  int F, kb, splits, batches, f_tiles, t_tiles, units;
  int w_rows_per_batch, x_cols_per_batch;  // batch offsets in the tensor maps' k coordinates
  float* out_f32;                          // [splits][T][F], or nullptr
  uint16_t* out_bf16;                      // out[t * out_ld + b * F + f], or nullptr
  int64_t out_ld;
};
struct GemmParams {
  GemmJob job[2];
  int njobs, T, total_units;
  int fsub;  // 128-feature blocks per unit: 2 (at most 128 tokens) or 1; token halves per unit: 3 - fsub
  unsigned long long wait_ns;  // bound of every wait (mla_sparse_set_wait_limit_ns)
};

struct GemmUnit {
  int j, b, ft, s, tt, k0, k1;
};
__device__ __forceinline__ GemmUnit unit_of(const GemmParams& p, int u) {
  GemmUnit g;
  g.j = (p.njobs > 1 && u >= p.job[0].units) ? 1 : 0;
  const GemmJob& J = p.job[g.j];
  int r = g.j ? u - p.job[0].units : u;
  g.s = r % J.splits;
  r /= J.splits;
  g.tt = r % J.t_tiles;
  r /= J.t_tiles;
  g.ft = r % J.f_tiles;
  g.b = r / J.f_tiles;
  g.k0 = g.s * J.kb / J.splits;
  g.k1 = (g.s + 1) * J.kb / J.splits;
  return g;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap w0, const __grid_constant__ CUtensorMap x0,
            const __grid_constant__ CUtensorMap w1, const __grid_constant__ CUtensorMap x1, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;  // the swizzled operands need 1024-byte alignment
  uint8_t* smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sb + kGemmOffBars + 8 * i; };
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(smem + kGemmOffBars + kGemmBars * 8);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kGemmOffBars + kGemmBars * 8 + 4);
  constexpr int kFull = 0, kEmpty = kGemmMaxStages, kAccFull = 2 * kGemmMaxStages, kAccEmpty = kAccFull + 2,
                kFinal = kAccEmpty + 2;
  constexpr int nst = kGemmMaxStages;
  // stage layout in 8 KB box units: weight boxes at 0 .. 2 fsub - 1 (A, two per
  // 128 features), token halves after them (B, two boxes of 64 rows each)
  const int fsub = p.fsub, tsub = 3 - p.fsub;
  const uint32_t kOffW = 0;
  const uint32_t kOffX = 2 * fsub * kBoxBytes;
  if (tid == 0) {
    *abort = 0u;
    for (int i = 0; i < kGemmMaxStages; ++i) {
      mbar_init(bar(kFull + i), 1);
      mbar_init(bar(kEmpty + i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(kAccFull + a), 1);
      mbar_init(bar(kAccEmpty + a), 128);
    }
    mbar_init(bar(kFinal), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
  // set-up done: the next launch of the chain may start its own; this grid's
  // inputs are complete once the previous launch of the chain has finished
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 4) {
    // TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        const GemmUnit g = unit_of(p, u);
        const GemmJob& J = p.job[g.j];
        const CUtensorMap* wm = g.j ? &w1 : &w0;
        const CUtensorMap* xm = g.j ? &x1 : &x0;
        const int f0 = g.ft * 128 * fsub, t0 = g.tt * 128 * tsub;
        const int nt = (tsub == 2 && t0 + 128 < p.T) ? 2 : 1;  // token halves loaded
        for (int kb = g.k0; kb < g.k1 && ok; ++kb, ++it) {
          const int st = it % nst;
          ok = mbar_wait<false>(bar(kEmpty + st), ((it / nst) & 1) ^ 1, abort, p.wait_ns);
          if (!ok) break;
          const uint32_t stage = sb + st * kGemmStageBytes;
          const uint32_t fb = bar(kFull + st);
          const int wk = g.b * J.w_rows_per_batch + kb * 64, xk = g.b * J.x_cols_per_batch + kb * 64;
          mbar_arrive_expect_tx(fb, (2 * fsub + 2 * nt) * kBoxBytes);
          for (int i = 0; i < 2 * fsub; ++i) tma_load_2d(stage + kOffW + i * kBoxBytes, wm, f0 + 64 * i, wk, fb);
          for (int h = 0; h < nt; ++h) tma_load_2d(stage + kOffX + 2 * h * kBoxBytes, xm, xk, t0 + 128 * h, fb);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_f16(128, 128, 1, 1, 0);
      constexpr uint32_t idesc256 = make_idesc_f16(128, 256, 1, 1, 0);
      int it = 0, lu = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x, ++lu) {
        const GemmUnit g = unit_of(p, u);
        const int nt = (tsub == 2 && g.tt * 256 + 128 < p.T) ? 2 : 1;
        const int a = lu & 1;
        ok = mbar_wait<false>(bar(kAccEmpty + a), ((lu >> 1) & 1) ^ 1, abort, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + 256 * a;
        for (int kb = g.k0; kb < g.k1; ++kb, ++it) {
          const int st = it % nst;
          ok = mbar_wait<false>(bar(kFull + st), (it / nst) & 1, abort, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t stage = sb + st * kGemmStageBytes;
          if (fsub == 1 && nt == 2) {
            // both 128-token halves in one N = 256 MMA: their boxes are contiguous
            // in the stage and their accumulator blocks (0, 0) and (0, 1) in TMEM
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_ss(d, make_sdesc(stage + kOffW + ks * 16 * 128, kBoxBytes, 1024, kSwizzle128B),
                      make_sdesc(stage + kOffX + ks * 32, 16, 1024, kSwizzle128B), idesc256,
                      (kb > g.k0 || ks > 0) ? 1u : 0u);
            umma_commit(bar(kEmpty + st));
            continue;
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t acc = (kb > g.k0 || ks > 0) ? 1u : 0u;
            // weight operand: k rows [16 ks, +16) of 128 features (two boxes, MN-major);
            // token operand: k columns [16 ks, +16) of 128 tokens (K-major); block (fs, h) at columns 128 (fs + h)
            for (int fs = 0; fs < fsub; ++fs) {
              const uint64_t wd =
                  make_sdesc(stage + kOffW + 2 * fs * kBoxBytes + ks * 16 * 128, kBoxBytes, 1024, kSwizzle128B);
              for (int h = 0; h < nt; ++h)
                umma_ss(d + 128 * (fs + h), wd,
                        make_sdesc(stage + kOffX + 2 * h * kBoxBytes + ks * 32, 16, 1024, kSwizzle128B), idesc, acc);
            }
          }
          umma_commit(bar(kEmpty + st));
        }
        if (!ok) break;
        umma_commit(bar(kAccFull + a));
      }
      umma_commit(bar(kFinal));
      volatile uint32_t never = 0;
      mbar_wait<false>(bar(kFinal), 0, &never, p.wait_ns > kGemmDrainNs ? p.wait_ns : kGemmDrainNs);
    }
    __syncwarp();
  } else {
    // epilogue: warp q reads TMEM lanes [32 q, +32)
    int lu = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++lu) {
      const GemmUnit g = unit_of(p, u);
      const GemmJob& J = p.job[g.j];
      const int a = lu & 1;
      if (!__all_sync(0xffffffffu, mbar_wait<false>(bar(kAccFull + a), (lu >> 1) & 1, abort, p.wait_ns))) break;
      tc_fence_after();
      const uint32_t lanes = static_cast<uint32_t>(32 * warp) << 16;
      {
        // lane = feature, columns = tokens; block (fs, h) at TMEM columns 128 (fs + h)
        for (int fs = 0; fs < fsub; ++fs) {
          const int f = (g.ft * fsub + fs) * 128 + 32 * warp + lane;
          const bool fin = f < J.F;
          for (int h = 0; h < tsub; ++h) {
            const int tb = g.tt * 128 * tsub + 128 * h;
            if (tb >= p.T) break;
#pragma unroll 1
            for (int ch = 0; ch < 4; ch += 2) {
              uint32_t v[64];  // two 32-token chunks per TMEM wait
              tmem_ld_32x32b_x32(tmem + lanes + 256 * a + 128 * (fs + h) + 32 * ch,
                                 *reinterpret_cast<uint32_t(*)[32]>(v));
              tmem_ld_32x32b_x32(tmem + lanes + 256 * a + 128 * (fs + h) + 32 * ch + 32,
                                 *reinterpret_cast<uint32_t(*)[32]>(v + 32));
              tmem_wait_ld();
              const int t0 = tb + 32 * ch;
              const int nv = p.T - t0;  // tokens of these chunks inside the call (>= 64: all)
              if (fin && nv > 0) {
                if (J.out_f32 != nullptr) {
                  float* o = J.out_f32 + (static_cast<int64_t>(g.s) * p.T + t0) * J.F + f;
                  if (nv >= 64) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) o[static_cast<int64_t>(k) * J.F] = __uint_as_float(v[k]);
                  } else {
#pragma unroll
                    for (int k = 0; k < 64; ++k)
                      if (k < nv) o[static_cast<int64_t>(k) * J.F] = __uint_as_float(v[k]);
                  }
                } else {
                  uint16_t* o = J.out_bf16 + static_cast<int64_t>(t0) * J.out_ld + static_cast<int64_t>(g.b) * J.F + f;
#pragma unroll
                  for (int k = 0; k < 64; ++k)
                    if (nv >= 64 || k < nv) {
                      const __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[k]));
                      o[static_cast<int64_t>(k) * J.out_ld] = *reinterpret_cast<const uint16_t*>(&hv);
                    }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kAccEmpty + a));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
  if (tid == 0 && *abort) atomicOr(&g_prolog_status, MLA_DEVICE_TIMEOUT);
}

// k-split counts: chosen from the shapes alone (the workspace size depends on
// them) so that the x projections have ~150 work units and the c^Q projection
// ~300; calls with many tokens have enough token tiles without splitting.
struct Splits {
  int x, b;
};
inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }
inline int fsub_of(int64_t T) { return T <= 128 ? 2 : 1; }
inline Splits splits_of(int64_t T, int64_t hidden, int64_t q_lora, int64_t H) {
  const int fw = 128 * fsub_of(T), tw = 128 * (3 - fsub_of(T));
  const int tt = ceil_div(T, tw);
  const int kbx = ceil_div(hidden, 64), kbb = ceil_div(q_lora, 64);
  const int fx = ceil_div(q_lora, fw) + ceil_div(kKv, fw);
  const int fb = ceil_div(H * kQHead, fw);
  Splits sp;
  sp.x = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kbx, 150 / (static_cast<int64_t>(fx) * tt))));
  sp.b = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(kbb, (300 + fb * tt / 2) / (static_cast<int64_t>(fb) * tt))));
  return sp;
}

struct Layout {
  size_t c_raw, kv_raw, c_q, q_raw, q_n, total;
  Splits sp;
};

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

inline Layout layout_of(int64_t T, int64_t hidden, int64_t q_lora, int64_t H) {
  Layout l;
  l.sp = splits_of(T, hidden, q_lora, H);
  size_t o = 0;
  l.c_raw = o;
  o = up256(o + size_t(l.sp.x) * size_t(T * q_lora) * 4);
  l.kv_raw = o;
  o = up256(o + size_t(l.sp.x) * size_t(T * kKv) * 4);
  l.c_q = o;
  o = up256(o + size_t(T * q_lora) * 2);
  l.q_raw = o;
  o = up256(o + size_t(l.sp.b) * size_t(T * H * kQHead) * 4);
  l.q_n = o;
  o = up256(o + size_t(T * H * kQkNope) * 2);
  l.total = o;
  return l;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_lock;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace mlapro

namespace {

thread_local char g_prolog_error[256] = "";

mla_status pro_fail(mla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mla_status pro_fail(mla_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_prolog_error, sizeof g_prolog_error, fmt, ap);
  va_end(ap);
  return s;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

bool dims_ok(const mla_prolog_dims* d) {
  return d && d->T >= 0 && d->hidden > 0 && d->hidden % 8 == 0 && d->q_lora > 0 && d->q_lora % 8 == 0 &&
         d->n_heads >= 1 && static_cast<int64_t>(d->T) * d->n_heads < (int64_t(1) << 31) &&
         static_cast<int64_t>(d->n_heads) * mlapro::kQHead < (int64_t(1) << 31) && d->num_rows >= 1 &&
         (d->kv_int8 == 0 || d->kv_int8 == 1) && d->eps > 0.f && d->eps < 1e30f;
}

#define PRO_CUDA(call, what)                                                                    \
  do {                                                                                          \
    const cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) return pro_fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

mla_status init_device(int dev, mlapro::DeviceState& st) {
  using namespace mlapro;
  if (st.ready) return MLA_OK;
  if (g_encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    PRO_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q),
             "looking up cuTensorMapEncodeTiled");
    if (q != cudaDriverEntryPointSuccess || fn == nullptr)
      return pro_fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  PRO_CUDA(cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem),
           "gemm kernel shared memory");
  PRO_CUDA(cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
  st.ready = true;
  return MLA_OK;
}

// Tensor map of a row-major bf16 matrix [rows, cols]: boxes of `box_rows` x
// 64 columns, 128-byte swizzle, zero fill outside.
mla_status tmap_2d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int box_rows, const char* what) {
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = mlapro::g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride,
                                      box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return pro_fail(MLA_ERR_CUDA, "tensor map of %s: error %d", what, static_cast<int>(r));
  return MLA_OK;
}

mlapro::GemmJob job_of(int64_t T, int F, int K, int splits, int batches, int rows_per_batch, int cols_per_batch,
                       float* out_f32, uint16_t* out_bf16, int64_t out_ld) {
  mlapro::GemmJob j;
  j.F = F;
  j.kb = mlapro::ceil_div(K, 64);
  j.splits = splits;
  j.batches = batches;
  j.f_tiles = mlapro::ceil_div(F, 128 * mlapro::fsub_of(T));
  j.t_tiles = mlapro::ceil_div(T, 128 * (3 - mlapro::fsub_of(T)));
  j.units = j.batches * j.f_tiles * j.splits * j.t_tiles;
  j.w_rows_per_batch = rows_per_batch;
  j.x_cols_per_batch = cols_per_batch;
  j.out_f32 = out_f32;
  j.out_bf16 = out_bf16;
  j.out_ld = out_ld;
  return j;
}

// Launch of one kernel of the call's chain on `s` as a programmatic dependent
// of the previous launch: its set-up overlaps the previous kernel's tail, and
// it waits (griddepcontrol.wait) for that kernel before reading its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

mla_status launch_gemm(const CUtensorMap& w0, const CUtensorMap& x0, const CUtensorMap& w1, const CUtensorMap& x1,
                       mlapro::GemmParams gp, int sms, cudaStream_t s, const char* what) {
  gp.total_units = gp.job[0].units + (gp.njobs > 1 ? gp.job[1].units : 0);
  gp.wait_ns = mlasp::host_wait_limit_ns();
  gp.fsub = mlapro::fsub_of(gp.T);
  const unsigned grid = static_cast<unsigned>(std::min(gp.total_units, sms));
  PRO_CUDA(launch_chained(mlapro::gemm_kernel, grid, mlapro::kGemmThreads, mlapro::kGemmSmem, s, w0, x0, w1, x1, gp),
           what);
  return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_prolog_workspace_bytes(const mla_prolog_dims* dims) {
  if (!dims_ok(dims)) return 0;
  return mlapro::layout_of(dims->T, dims->hidden, dims->q_lora, dims->n_heads).total;
}

mla_status mla_prolog(const mla_prolog_dims* dims, const void* x, const mla_prolog_weights* w, const float* cos,
                      const float* sin, const int64_t* cache_index, void* q_nope, void* q_rope, void* kv_nope,
                      void* kv_rope, float* kv_scales, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace mlapro;
  g_prolog_error[0] = '\0';
  if (!dims) return pro_fail(MLA_ERR_NULL, "dims is NULL");
  if (!dims_ok(dims))
    return pro_fail(MLA_ERR_SHAPE,
                    "T=%d hidden=%d q_lora=%d n_heads=%d num_rows=%lld kv_int8=%d eps=%g: hidden and q_lora must be "
                    "positive multiples of 8, n_heads >= 1, T * n_heads < 2^31, num_rows >= 1, eps > 0",
                    dims->T, dims->hidden, dims->q_lora, dims->n_heads, static_cast<long long>(dims->num_rows),
                    dims->kv_int8, static_cast<double>(dims->eps));
  if (dims->T == 0) return MLA_OK;  // nothing is read or written
  if (!x || !w || !cos || !sin || !cache_index || !q_nope || !q_rope || !kv_nope || !kv_rope || !workspace ||
      (dims->kv_int8 && !kv_scales))
    return pro_fail(MLA_ERR_NULL, "a required pointer is NULL");
  if (!w->wq_a || !w->gamma_cq || !w->wq_b || !w->w_uk || !w->wkv || !w->gamma_ckv)
    return pro_fail(MLA_ERR_NULL, "a weight pointer is NULL");
  const void* p16[] = {x, w->wq_a, w->gamma_cq, w->wq_b, w->w_uk, w->wkv, w->gamma_ckv, cos, sin,
                       q_nope, q_rope, kv_nope, kv_rope};
  for (const void* ptr : p16)
    if (!aligned(ptr, 16)) return pro_fail(MLA_ERR_ALIGN, "tensors must be 16-byte aligned");
  if ((dims->kv_int8 && !aligned(kv_scales, 16)) || !aligned(cache_index, 8) || !aligned(workspace, 256))
    return pro_fail(MLA_ERR_ALIGN, "kv_scales 16-byte, cache_index 8-byte and workspace 256-byte alignment");
  const int T = dims->T, H = dims->n_heads, hidden = dims->hidden, q_lora = dims->q_lora;
  const Layout L = layout_of(T, hidden, q_lora, H);
  if (workspace_bytes < L.total)
    return pro_fail(MLA_ERR_SHAPE, "workspace of %zu bytes, %zu needed", workspace_bytes, L.total);
  int dev = 0;
  PRO_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return pro_fail(MLA_ERR_UNSUPPORTED, "device %d", dev);

  int sms = 0;
  {
    std::lock_guard<std::mutex> guard(g_lock);
    DeviceState& st = g_dev[dev];
    const mla_status ist = init_device(dev, st);
    if (ist != MLA_OK) return ist;
    sms = st.sms;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* c_raw = reinterpret_cast<float*>(ws + L.c_raw);
  float* kv_raw = reinterpret_cast<float*>(ws + L.kv_raw);
  uint16_t* c_q = reinterpret_cast<uint16_t*>(ws + L.c_q);
  float* q_raw = reinterpret_cast<float*>(ws + L.q_raw);
  uint16_t* q_n = reinterpret_cast<uint16_t*>(ws + L.q_n);

  NormParams np;
  np.c_raw = c_raw;
  np.gamma_cq = static_cast<const uint16_t*>(w->gamma_cq);
  np.c_q = c_q;
  np.kv_raw = kv_raw;
  np.gamma_ckv = static_cast<const uint16_t*>(w->gamma_ckv);
  np.cos = cos;
  np.sin = sin;
  np.idx = cache_index;
  np.kv_nope = static_cast<uint8_t*>(kv_nope);
  np.kv_rope = static_cast<uint8_t*>(kv_rope);
  np.kv_scales = kv_scales;
  np.num_rows = dims->num_rows;
  np.q_lora = q_lora;
  np.T = T;
  np.int8 = dims->kv_int8;
  np.c_slots = L.sp.x;
  np.kv_slots = L.sp.x;
  np.eps = dims->eps;

  HeadParams hp;
  hp.q_raw = q_raw;
  hp.cos = cos;
  hp.sin = sin;
  hp.q_n = q_n;
  hp.q_rope = static_cast<uint16_t*>(q_rope);
  hp.H = H;
  hp.TH = T * H;
  hp.q_slots = L.sp.b;
  hp.eps = dims->eps;

  // tensor maps: weights [K rows, F columns] in boxes of 64 x 64, token operands [T, K] in boxes of 128 x 64
  CUtensorMap m_x, m_wqa, m_wkv, m_cq, m_wqb, m_qn, m_wuk;
  mla_status ms = tmap_2d(&m_x, x, hidden, T, 128, "x");
  if (ms == MLA_OK) ms = tmap_2d(&m_wqa, w->wq_a, q_lora, hidden, 64, "wq_a");
  if (ms == MLA_OK) ms = tmap_2d(&m_wkv, w->wkv, kKv, hidden, 64, "wkv");
  if (ms == MLA_OK) ms = tmap_2d(&m_cq, c_q, q_lora, T, 128, "c^Q");
  if (ms == MLA_OK) ms = tmap_2d(&m_wqb, w->wq_b, static_cast<int64_t>(H) * kQHead, q_lora, 64, "wq_b");
  if (ms == MLA_OK) ms = tmap_2d(&m_qn, q_n, static_cast<int64_t>(H) * kQkNope, T, 128, "q");
  if (ms == MLA_OK) ms = tmap_2d(&m_wuk, w->w_uk, kLatent, static_cast<int64_t>(H) * kQkNope, 64, "w_uk");
  if (ms != MLA_OK) return ms;

  // x @ wq_a and x @ wkv side by side in one launch
  GemmParams gx;
  gx.njobs = 2;
  gx.T = T;
  gx.job[0] = job_of(T, q_lora, hidden, L.sp.x, 1, 0, 0, c_raw, nullptr, 0);
  gx.job[1] = job_of(T, kKv, hidden, L.sp.x, 1, 0, 0, kv_raw, nullptr, 0);
  ms = launch_gemm(m_wqa, m_x, m_wkv, m_x, gx, sms, s, "x projections launch");
  if (ms != MLA_OK) return ms;
  np.c_slots = L.sp.x;
  np.kv_slots = L.sp.x;
  const size_t row_smem = q_lora <= kStageCqMax ? static_cast<size_t>(q_lora) * 4 : 0;
  PRO_CUDA(launch_chained(x_rows_kernel, static_cast<unsigned>(T), kRowThreads, row_smem, s, np), "x_rows_kernel launch");
  // c^Q @ wq_b
  GemmParams gb;
  gb.njobs = 1;
  gb.T = T;
  gb.job[0] = job_of(T, H * kQHead, q_lora, L.sp.b, 1, 0, 0, q_raw, nullptr, 0);
  gb.job[1] = gb.job[0];
  ms = launch_gemm(m_wqb, m_cq, m_wqb, m_cq, gb, sms, s, "c^Q projection launch");
  if (ms != MLA_OK) return ms;
  PRO_CUDA(launch_chained(q_heads_kernel, static_cast<unsigned>((static_cast<int64_t>(T) * H + kWarps - 1) / kWarps),
                          kWarps * 32, 0, s, hp),
           "q_heads_kernel launch");
  // absorption: head h, q_nope[:, h, :] (row stride H * 512) = q[:, h, :128] @ w_uk[h]
  GemmParams ga;
  ga.njobs = 1;
  ga.T = T;
  ga.job[0] = job_of(T, kLatent, kQkNope, 1, H, kQkNope, kQkNope, nullptr, static_cast<uint16_t*>(q_nope),
                     static_cast<int64_t>(H) * kLatent);
  ga.job[1] = ga.job[0];
  return launch_gemm(m_wuk, m_qn, m_wuk, m_qn, ga, sms, s, "absorption launch");
}

const char* mla_prolog_last_error(void) { return g_prolog_error; }

mla_status mla_prolog_device_status(void* stream, uint32_t* flags, int32_t clear) {
  g_prolog_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pro_fail(MLA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, mlapro::g_prolog_status, sizeof v);
  if (e != cudaSuccess) return pro_fail(MLA_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(mlapro::g_prolog_status, &zero, sizeof zero);
    if (e != cudaSuccess) return pro_fail(MLA_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  if (flags) *flags = v;
  if (v != 0) return pro_fail(MLA_ERR_DEVICE_STATUS, "prolog device status 0x%x", v);
  return MLA_OK;
}

}  // extern "C"
