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
// Data flow per call (T tokens, H heads), seven launches:
//   side stream   kv_raw = x @ wkv                     cuBLAS, fp32 out
//   side stream   kv_rows_kernel: k = RMSNorm(kv_raw) * gamma_ckv, RoPE on
//                 k[512:], rounded to bf16 and written (bf16 or INT8) into
//                 the cache row
//   stream        c_raw  = x @ wq_a                    cuBLAS, fp32 out
//   stream        cq_rows_kernel: c^Q = bf16(RMSNorm(c_raw) * gamma_cq)
//   stream        q_raw  = c^Q @ wq_b                  cuBLAS, fp32 out
//   stream        q_heads_kernel: per (t, h) RMSNorm over 192, q[:128] -> bf16
//                 operand, RoPE(q[128:]) -> q_rope
//   stream        q_nope[h] = q[h][:128] @ w_uk[h]     cuBLAS strided batched, bf16 out
//   stream        waits for the side stream
// The query and key paths are independent after x (the page runs the two
// projections side by side because neither fills the machine in decode);
// here they run on two streams.  The norms are memory-bound row passes in
// fp32 with one rounding to bf16 at each storage point: a 128-thread block
// per c^Q row, a warp per key row and per (token, head).
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "../../include/mla_prolog.h"

namespace mlapro {

constexpr int kWarps = 8;
constexpr int kQkNope = 128;
constexpr int kRope = 64;
constexpr int kLatent = 512;
constexpr int kKv = kLatent + kRope;  // 576
constexpr int kQHead = kQkNope + kRope;  // 192
constexpr size_t kBlasWsMain = size_t(32) << 20;
constexpr size_t kBlasWsSide = size_t(8) << 20;

__device__ unsigned int g_prolog_status = 0;

struct NormParams {
  const float* c_raw;        // [T, q_lora]
  const uint16_t* gamma_cq;  // bf16 [q_lora]
  uint16_t* c_q;             // bf16 [T, q_lora]
  const float* kv_raw;       // [T, 576]
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
  float eps;
};

struct HeadParams {
  const float* q_raw;  // [T * H, 192]
  const float* cos;
  const float* sin;
  uint16_t* q_n;       // bf16 [T * H, 128]
  uint16_t* q_rope;    // bf16 [T * H, 64]
  int H;
  int TH;
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

constexpr int kCqThreads = 128;

// One block per c^Q row: sum of squares over the row, then the scaled, rounded row.
__global__ void __launch_bounds__(kCqThreads) cq_rows_kernel(const NormParams p) {
  __shared__ float part[kCqThreads / 32];
  const int t = blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(p.c_raw + static_cast<int64_t>(t) * p.q_lora);
  const int n4 = p.q_lora >> 2;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += kCqThreads) {
    const float4 v = src[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCqThreads / 32; ++w) tot += part[w];
  const float inv = inv_rms(tot, p.q_lora, p.eps);
  const uint2* gam = reinterpret_cast<const uint2*>(p.gamma_cq);
  uint2* dst = reinterpret_cast<uint2*>(p.c_q + static_cast<int64_t>(t) * p.q_lora);
  for (int i = threadIdx.x; i < n4; i += kCqThreads) {
    const float4 v = src[i];
    const uint2 gw = __ldg(gam + i);
    dst[i] = make_uint2(pack_bf16(v.x * inv * bf16_lo(gw.x), v.y * inv * bf16_hi(gw.x)),
                        pack_bf16(v.z * inv * bf16_lo(gw.y), v.w * inv * bf16_hi(gw.y)));
  }
}

// One warp per key row: RMSNorm over the 576-wide row, RoPE on its tail, the cache write.
__global__ void __launch_bounds__(kWarps * 32) kv_rows_kernel(const NormParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= p.T) return;
  // lane l: latent dims [16 l, 16 l + 16) (eight lanes per 128-element group) and rope pair l
  const float* row = p.kv_raw + static_cast<int64_t>(t) * kKv;
  float x[16];
  {
    const float4* s4 = reinterpret_cast<const float4*>(row + 16 * lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 v = s4[k];
      x[4 * k] = v.x;
      x[4 * k + 1] = v.y;
      x[4 * k + 2] = v.z;
      x[4 * k + 3] = v.w;
    }
  }
  const float2 rp = reinterpret_cast<const float2*>(row + kLatent)[lane];
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

// One warp per (token, head): lane l holds dims (2l, 2l+1), (64+2l, 65+2l) and rope pair l.
__global__ void __launch_bounds__(kWarps * 32) q_heads_kernel(const HeadParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kWarps + warp;
  if (g >= p.TH) return;
  const int t = g / p.H;
  const float2* row = reinterpret_cast<const float2*>(p.q_raw + static_cast<int64_t>(g) * kQHead);
  const float2 u = row[lane], v = row[32 + lane], w = row[64 + lane];
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

struct Layout {
  size_t c_raw, kv_raw, c_q, q_raw, q_n, ws_main, ws_side, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

inline Layout layout_of(int64_t T, int64_t q_lora, int64_t H) {
  Layout l;
  size_t o = 0;
  l.c_raw = o;
  o = up256(o + size_t(T * q_lora) * 4);
  l.kv_raw = o;
  o = up256(o + size_t(T * kKv) * 4);
  l.c_q = o;
  o = up256(o + size_t(T * q_lora) * 2);
  l.q_raw = o;
  o = up256(o + size_t(T * H * kQHead) * 4);
  l.q_n = o;
  o = up256(o + size_t(T * H * kQkNope) * 2);
  l.ws_main = o;
  o = up256(o + kBlasWsMain);
  l.ws_side = o;
  o = up256(o + kBlasWsSide);
  l.total = o;
  return l;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  cublasHandle_t blas = nullptr;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_lock;

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

#define PRO_BLAS(call, what)                                                                            \
  do {                                                                                                  \
    const cublasStatus_t s_ = (call);                                                                   \
    if (s_ != CUBLAS_STATUS_SUCCESS) return pro_fail(MLA_ERR_CUDA, "%s: %s", what, cublasGetStatusString(s_)); \
  } while (0)

mla_status init_device(mlapro::DeviceState& st) {
  if (st.ready) return MLA_OK;
  PRO_BLAS(cublasCreate(&st.blas), "cublasCreate");
  PRO_BLAS(cublasSetMathMode(st.blas, static_cast<cublasMath_t>(CUBLAS_DEFAULT_MATH |
                                                                CUBLAS_MATH_DISALLOW_REDUCED_PRECISION_REDUCTION)),
           "cublasSetMathMode");
  PRO_CUDA(cudaStreamCreateWithFlags(&st.side, cudaStreamNonBlocking), "creating the side stream");
  PRO_CUDA(cudaEventCreateWithFlags(&st.fork, cudaEventDisableTiming), "creating an event");
  PRO_CUDA(cudaEventCreateWithFlags(&st.join, cudaEventDisableTiming), "creating an event");
  st.ready = true;
  return MLA_OK;
}

// Row-major C[M, N] (fp32 or bf16) = A[M, K] @ B[K, N] (bf16), as cuBLAS's column-major C^T = B^T A^T.
mla_status gemm_rm(cublasHandle_t h, int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C,
                   int ldc, cudaDataType_t c_type, const char* what) {
  const float one = 1.f, zero = 0.f;
  PRO_BLAS(cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, N, M, K, &one, B, CUDA_R_16BF, ldb, A, CUDA_R_16BF, lda, &zero, C,
                        c_type, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
           what);
  return MLA_OK;
}

}  // namespace

extern "C" {

size_t mla_prolog_workspace_bytes(const mla_prolog_dims* dims) {
  if (!dims_ok(dims)) return 0;
  return mlapro::layout_of(dims->T, dims->q_lora, dims->n_heads).total;
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
  const Layout L = layout_of(T, q_lora, H);
  if (workspace_bytes < L.total)
    return pro_fail(MLA_ERR_SHAPE, "workspace of %zu bytes, %zu needed", workspace_bytes, L.total);
  int dev = 0;
  PRO_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return pro_fail(MLA_ERR_UNSUPPORTED, "device %d", dev);

  std::lock_guard<std::mutex> guard(g_lock);
  DeviceState& st = g_dev[dev];
  const mla_status ist = init_device(st);
  if (ist != MLA_OK) return ist;
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
  np.eps = dims->eps;

  HeadParams hp;
  hp.q_raw = q_raw;
  hp.cos = cos;
  hp.sin = sin;
  hp.q_n = q_n;
  hp.q_rope = static_cast<uint16_t*>(q_rope);
  hp.H = H;
  hp.TH = T * H;
  hp.eps = dims->eps;

  // key path on the side stream, forked from `s` here; whatever the paths enqueue, the side stream is
  // joined back into `s` before returning, also when a step fails part-way
  PRO_CUDA(cudaEventRecord(st.fork, s), "recording the fork event");
  PRO_CUDA(cudaStreamWaitEvent(st.side, st.fork, 0), "side stream wait");
  auto paths = [&]() -> mla_status {
    PRO_BLAS(cublasSetStream(st.blas, st.side), "cublasSetStream");
    PRO_BLAS(cublasSetWorkspace(st.blas, ws + L.ws_side, kBlasWsSide), "cublasSetWorkspace");
    mla_status gs = gemm_rm(st.blas, T, kKv, hidden, x, hidden, w->wkv, kKv, kv_raw, kKv, CUDA_R_32F, "x @ wkv");
    if (gs != MLA_OK) return gs;
    kv_rows_kernel<<<static_cast<unsigned>((T + kWarps - 1) / kWarps), kWarps * 32, 0, st.side>>>(np);
    PRO_CUDA(cudaGetLastError(), "kv_rows_kernel launch");

    // query path on `s`
    PRO_BLAS(cublasSetStream(st.blas, s), "cublasSetStream");
    PRO_BLAS(cublasSetWorkspace(st.blas, ws + L.ws_main, kBlasWsMain), "cublasSetWorkspace");
    gs = gemm_rm(st.blas, T, q_lora, hidden, x, hidden, w->wq_a, q_lora, c_raw, q_lora, CUDA_R_32F, "x @ wq_a");
    if (gs != MLA_OK) return gs;
    cq_rows_kernel<<<static_cast<unsigned>(T), kCqThreads, 0, s>>>(np);
    PRO_CUDA(cudaGetLastError(), "cq_rows_kernel launch");
    gs = gemm_rm(st.blas, T, H * kQHead, q_lora, c_q, q_lora, w->wq_b, H * kQHead, q_raw, H * kQHead, CUDA_R_32F,
                 "c^Q @ wq_b");
    if (gs != MLA_OK) return gs;
    q_heads_kernel<<<static_cast<unsigned>((static_cast<int64_t>(T) * H + kWarps - 1) / kWarps), kWarps * 32, 0,
                     s>>>(hp);
    PRO_CUDA(cudaGetLastError(), "q_heads_kernel launch");
    // absorption: head h, C_h[T, 512] (row stride H * 512) = q_n[:, h] [T, 128] (row stride H * 128) @ w_uk[h]
    const float one = 1.f, zero = 0.f;
    PRO_BLAS(cublasGemmStridedBatchedEx(st.blas, CUBLAS_OP_N, CUBLAS_OP_N, kLatent, T, kQkNope, &one, w->w_uk,
                                        CUDA_R_16BF, kLatent, static_cast<long long>(kQkNope) * kLatent, q_n,
                                        CUDA_R_16BF, H * kQkNope, kQkNope, &zero, q_nope, CUDA_R_16BF, H * kLatent,
                                        kLatent, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
             "absorption q_nope @ w_uk");
    return MLA_OK;
  };
  const mla_status body = paths();
  cudaError_t ej = cudaEventRecord(st.join, st.side);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, st.join, 0);
  if (body != MLA_OK) return body;  // its message stands
  if (ej != cudaSuccess) return pro_fail(MLA_ERR_CUDA, "joining the side stream: %s", cudaGetErrorString(ej));
  return MLA_OK;
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
