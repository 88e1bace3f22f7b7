// Paged MLA cache writer for GB300 (sm_103a): new key rows into the bf16 or
// INT8 cache that the sparse attention kernel reads.
//
// Layout and INT8 rule: "DeepSeek V3/V2 Sparse Flash Attention with
// Quantization" (operator spec, inputs/outputs, quantisation note); the write
// at cache_index is the cache-update step of MlaProlog ("NPU DeepSeek-V4 PyPTO
// fused-operator optimization").  One warp per new row: lane l holds latent
// dims [16 l, 16 l + 16), so the eight lanes of a 128-element group find its
// absolute maximum with three shuffles; lanes 0-7 also copy the 128-byte rope
// row.  HBM-bound and tiny per call; one launch.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/mla_cache.h"

namespace mlacw {

constexpr int kWarps = 8;

__device__ unsigned int g_cache_status = 0;

struct Params {
  const uint8_t* k_nope;  // bf16 [T, 512]
  const uint8_t* k_rope;  // bf16 [T, 64]
  const int64_t* idx;
  uint8_t* kv_nope;
  uint8_t* kv_rope;
  float* kv_scales;
  int64_t num_rows;
  int T;
  int int8;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round half to even of x / scale (fp32 division, correctly rounded), clamped.
__device__ __forceinline__ uint32_t code8(float x, float scale) {
  const int q = __float2int_rn(__fdiv_rn(x, scale));
  return static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(max(-128, min(127, q)))));
}

__global__ void __launch_bounds__(kWarps * 32) cache_write_kernel(const Params p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= p.T) return;
  // The new row does not depend on its index: both loads are in flight together.
  const uint4* src = reinterpret_cast<const uint4*>(p.k_nope + static_cast<int64_t>(t) * 1024) + 2 * lane;
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  const uint4 rope = __ldg(reinterpret_cast<const uint4*>(p.k_rope + static_cast<int64_t>(t) * 128) + (lane & 7));
  const int64_t r = __ldg(p.idx + t);
  if (r < 0) return;
  if (r >= p.num_rows) {
    if (lane == 0) atomicOr(&g_cache_status, MLA_DEVICE_BAD_BLOCK);
    return;
  }
  if (lane < 8) reinterpret_cast<uint4*>(p.kv_rope + r * 128)[lane] = rope;
  if (!p.int8) {
    uint4* dst = reinterpret_cast<uint4*>(p.kv_nope + r * 1024) + 2 * lane;
    dst[0] = a;
    dst[1] = b;
    return;
  }
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[2 * k] = bf16_lo(w[k]);
    x[2 * k + 1] = bf16_hi(w[k]);
  }
  float am = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) am = fmaxf(am, fabsf(x[k]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  float scale = __fdiv_rn(am, 127.f);
  if (!(scale > 0.f)) scale = 1.f;
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    c[k] = code8(x[4 * k], scale) | (code8(x[4 * k + 1], scale) << 8) | (code8(x[4 * k + 2], scale) << 16) |
           (code8(x[4 * k + 3], scale) << 24);
  reinterpret_cast<uint4*>(p.kv_nope + r * 512)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
  if ((lane & 7) == 0) p.kv_scales[r * 4 + (lane >> 3)] = scale;
}

}  // namespace mlacw

namespace {

thread_local char g_cache_error[256] = "";

mla_status cache_fail(mla_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mla_status cache_fail(mla_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_cache_error, sizeof g_cache_error, fmt, ap);
  va_end(ap);
  return s;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace

extern "C" {

mla_status mla_cache_write(int32_t T, int64_t num_rows, int32_t kv_int8, const void* k_nope, const void* k_rope,
                           const int64_t* cache_index, void* kv_nope, void* kv_rope, float* kv_scales,
                           void* stream) {
  g_cache_error[0] = '\0';
  if (T < 0 || num_rows < 1) return cache_fail(MLA_ERR_SHAPE, "T=%d num_rows=%lld", T, static_cast<long long>(num_rows));
  if (kv_int8 != 0 && kv_int8 != 1) return cache_fail(MLA_ERR_SHAPE, "kv_int8=%d must be 0 or 1", kv_int8);
  if (T == 0) return MLA_OK;  // nothing is read or written; empty arrays may have null pointers
  if (!k_nope || !k_rope || !cache_index || !kv_nope || !kv_rope || (kv_int8 && !kv_scales))
    return cache_fail(MLA_ERR_NULL, "a required pointer is NULL");
  if (!aligned(k_nope, 16) || !aligned(k_rope, 16) || !aligned(kv_nope, 16) || !aligned(kv_rope, 16) ||
      (kv_int8 && !aligned(kv_scales, 16)) || !aligned(cache_index, 8))
    return cache_fail(MLA_ERR_ALIGN, "rows and caches must be 16-byte aligned, cache_index 8-byte");
  mlacw::Params p;
  p.k_nope = static_cast<const uint8_t*>(k_nope);
  p.k_rope = static_cast<const uint8_t*>(k_rope);
  p.idx = cache_index;
  p.kv_nope = static_cast<uint8_t*>(kv_nope);
  p.kv_rope = static_cast<uint8_t*>(kv_rope);
  p.kv_scales = kv_scales;
  p.num_rows = num_rows;
  p.T = T;
  p.int8 = kv_int8;
  const unsigned grid = static_cast<unsigned>((T + mlacw::kWarps - 1) / mlacw::kWarps);
  mlacw::cache_write_kernel<<<grid, mlacw::kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cache_fail(MLA_ERR_CUDA, "cache write launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}

const char* mla_cache_last_error(void) { return g_cache_error; }

mla_status mla_cache_device_status(void* stream, uint32_t* flags, int32_t clear) {
  g_cache_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cache_fail(MLA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, mlacw::g_cache_status, sizeof v);
  if (e != cudaSuccess) return cache_fail(MLA_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(mlacw::g_cache_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cache_fail(MLA_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  if (flags) *flags = v;
  if (v != 0) return cache_fail(MLA_ERR_DEVICE_STATUS, "cache writer device status 0x%x", v);
  return MLA_OK;
}

}  // extern "C"
