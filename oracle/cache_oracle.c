/*
 * TEST INFRASTRUCTURE ONLY -- the oracle for writing new key rows into the
 * paged MLA cache (bf16, or INT8 with fp32 group scales).  Only tests/, the
 * smoke check and the benchmark's CPU-baseline leg may load this library; the
 * product path never calls it and shares no code with it.
 *
 * Written from "DeepSeek V3/V2 Sparse Flash Attention with Quantization":
 *   - section "算子规格" / "输入输出" (operator spec, inputs/outputs): the cache
 *     is key_nope_2d (rows, 512) BF16 or INT8, key_rope_2d (rows, 64) BF16 and
 *     k_nope_scales (rows, 4) FP32, one scale per 128 elements, rows =
 *     block_num * block_size;
 *   - section "注意事项" (notes), INT8 quantisation rule: the nope part is split
 *     into groups of 128 elements; each group's absolute maximum sets the
 *     scale and the values are quantised into [-128, 127];
 * and from "NPU DeepSeek-V4 PyPTO fused-operator optimization", section
 * MlaProlog, whose operator writes the new k rows into the cache at
 * cache_index.
 * Readings where the pages are open:
 *   - cache_index[t] is the flat physical row (block id * block_size + offset)
 *     that new row t goes to; a negative index means "no row" and is skipped;
 *     an index at or beyond the cache's row count is skipped and counted;
 *   - scale = absmax / 127 in fp32 (so that the extreme element maps to
 *     +-127); a group whose scale is not positive (all zeros, or an absmax so
 *     small that absmax / 127 underflows) gets scale 1;
 *   - code = clamp(round_half_even(x / scale), -128, 127), the division and
 *     the rounding in fp32 (the precision the kernel decides the code in);
 *   - rows are written independently; indices are expected to be distinct.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float cw_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * k_nope (T, 512) and k_rope (T, 64) as bf16 bits.  kv_nope is uint16 (bf16)
 * when kv_int8 == 0, else int8 with kv_scales (rows, 4) fp32.  Returns 0, or
 * -1 on bad arguments; *skipped_bad counts indices at or beyond num_rows.
 */
int cache_oracle_write(int T, int kv_int8, int64_t num_rows, const uint16_t* k_nope, const uint16_t* k_rope,
                       const int64_t* cache_index, void* kv_nope, uint16_t* kv_rope, float* kv_scales,
                       int64_t* skipped_bad) {
  if (T < 0 || num_rows <= 0 || (kv_int8 && kv_scales == NULL)) return -1;
  int64_t bad = 0;
  for (int t = 0; t < T; ++t) {
    const int64_t r = cache_index[t];
    if (r < 0) continue;
    if (r >= num_rows) {
      ++bad;
      continue;
    }
    memcpy(kv_rope + r * 64, k_rope + (int64_t)t * 64, 64 * sizeof(uint16_t));
    const uint16_t* x = k_nope + (int64_t)t * 512;
    if (!kv_int8) {
      memcpy((uint16_t*)kv_nope + r * 512, x, 512 * sizeof(uint16_t));
      continue;
    }
    int8_t* q = (int8_t*)kv_nope + r * 512;
    for (int g = 0; g < 4; ++g) {
      float absmax = 0.0f;
      for (int i = 0; i < 128; ++i) {
        const float a = fabsf(cw_bf16(x[g * 128 + i]));
        if (a > absmax) absmax = a;
      }
      float scale = absmax / 127.0f;
      if (!(scale > 0.0f)) scale = 1.0f;
      for (int i = 0; i < 128; ++i) {
        const float v = rintf(cw_bf16(x[g * 128 + i]) / scale); /* round half to even (default mode) */
        q[g * 128 + i] = (int8_t)(v > 127.0f ? 127.0f : (v < -128.0f ? -128.0f : v));
      }
      kv_scales[r * 4 + g] = scale;
    }
  }
  if (skipped_bad) *skipped_bad = bad;
  return 0;
}
