/*
 * TEST INFRASTRUCTURE ONLY -- the oracle.  Only tests/, the smoke check and
 * the benchmark's CPU-baseline leg may load this library; the product path
 * never calls it and shares no code with it.
 *
 * Plain, slow, obviously-correct fp64 CPU definition of DeepSeek-style MLA
 * sparse attention over a paged KV cache, written from:
 *   - "DeepSeek V3/V2 Sparse Flash Attention with Quantization"
 *     (sparse_flash_attention_quant): section "Algorithm overview" (MLA split
 *     into a 512-dim nope part and a 64-dim rope part, top-k sparse
 *     selection, INT8 KV cache in groups of 128 with one FP32 scale, paged
 *     cache with block_size 128 and block_table, per-batch actual length),
 *     section "Inputs / outputs" (tensor shapes), section "INT8 quantization
 *     path" (INT8 -> FP16 -> FP32, times the group scale, -> BF16), and
 *     section "Decode mode" (softmax = exp(S - max S) / sum exp(S - max S));
 *   - "CANN DeepSeek Indexer attention", section "Sparse Flash Attention"
 *     (o_i = Attn(x_i, {c_j : j in Top-k(I_i,:)})).
 *
 * For each query token t = (b, s) and query head h:
 *   1. valid entries: i with 0 <= topk[t,i] < act_seq[b] (a multiset over the
 *      list: a repeated index counts once per occurrence);
 *   2. physical row r_i = block_table[b, j / block_size] * block_size
 *      + j % block_size for j = topk[t,i]; a block id outside
 *      [0, num_blocks), or a table slot j / block_size beyond the table's
 *      width, makes the entry invalid (the CUDA path masks it the same way
 *      and raises a status bit);
 *   3. z_i = scale * (sum_d qn[t,h,d] Kn[r_i,d] + sum_d qr[t,h,d] Kr[r_i,d]);
 *   4. m = max z, l = sum exp(z_i - m);
 *   5. out[t,h,:] = sum exp(z_i - m) Kn[r_i,:] / l;  lse[t,h] = m + ln l.
 * With no valid entry: out = 0, lse = -inf.
 *
 * Inputs are widened exactly from bf16.  INT8 rows are dequantised as the
 * INT8 path prescribes: the FP32 product (float)q8 * scale, rounded to BF16
 * (round to nearest even), then widened exactly.  Everything after that is
 * fp64.  No online softmax, no tiling: the prefill algorithm is a reordering
 * of this same sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp32 -> bf16 bits, round to nearest, ties to even; NaN stays NaN. */
static uint16_t float_to_bf16_bits_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* INT8 path: INT8 -> FP16 -> FP32 (both exact), times the FP32 group scale
 * (one FP32 rounding), then to BF16. */
uint16_t mla_oracle_dequant_bits(int8_t q, float scale) {
  volatile float prod = (float)q * scale; /* volatile: keep it one fp32 multiply */
  return float_to_bf16_bits_rne(prod);
}

void mla_oracle_dequant_rows(const int8_t* q, const float* scales, int64_t rows, int d_nope,
                             uint16_t* out_bf16) {
  const int groups = d_nope / 128;
  for (int64_t r = 0; r < rows; ++r)
    for (int d = 0; d < d_nope; ++d)
      out_bf16[r * d_nope + d] = mla_oracle_dequant_bits(q[r * d_nope + d], scales[r * groups + d / 128]);
}

/*
 * Returns 0 on success, a negative value on bad arguments.
 * tokens: list of n_tokens token ids to evaluate (NULL: all B*S1 tokens in
 * order).  out: (n_tokens, n_q, d_nope) fp64.  lse: (n_tokens, n_q) fp64.
 * bad_blocks (may be NULL): receives the number of valid entries whose
 * block id was outside [0, num_blocks).
 */
int mla_oracle_fwd(int B, int S1, int n_q, int n_kv, int d_nope, int d_rope, int block_size,
                   int num_blocks, int max_blocks_per_seq, int topk, int kv_int8,
                   const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_nope,
                   const uint16_t* kv_rope, const float* kv_scales, const int32_t* topk_idx,
                   const int32_t* block_table, const int32_t* act_seqs, double softmax_scale,
                   const int32_t* tokens, int n_tokens, double* out, double* lse, int n_threads,
                   int64_t* bad_blocks) {
  if (B <= 0 || S1 <= 0 || n_q <= 0 || n_kv != 1 || d_nope <= 0 || d_rope < 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0 || topk <= 0)
    return -1;
  if (kv_int8 && (d_nope % 128 != 0 || kv_scales == NULL)) return -2;
  const int T = B * S1;
  if (tokens == NULL) n_tokens = T;
  const int D = d_nope + d_rope;
  int64_t bad_total = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads) reduction(+ : bad_total)
#endif
  {
    double* K = (double*)malloc(sizeof(double) * (size_t)topk * (size_t)D);
    double* z = (double*)malloc(sizeof(double) * (size_t)topk);
    double* q = (double*)malloc(sizeof(double) * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int n = 0; n < n_tokens; ++n) {
      const int t = tokens ? tokens[n] : n;
      const int b = t / S1;
      const int act = act_seqs[b];
      /* steps 1-2: the valid entries and their rows, widened once */
      int nv = 0;
      for (int i = 0; i < topk; ++i) {
        const int j = topk_idx[(int64_t)t * topk + i];
        if (j < 0 || j >= act) continue;
        const int blk_slot = j / block_size;
        const int blk = blk_slot < max_blocks_per_seq ? block_table[(int64_t)b * max_blocks_per_seq + blk_slot] : -1;
        if (blk < 0 || blk >= num_blocks) {
          ++bad_total;
          continue;
        }
        const int64_t r = (int64_t)blk * block_size + j % block_size;
        double* row = K + (size_t)nv * D;
        for (int d = 0; d < d_nope; ++d) {
          if (kv_int8) {
            const int8_t q8 = ((const int8_t*)kv_nope)[r * d_nope + d];
            row[d] = bf16_bits_to_double(mla_oracle_dequant_bits(q8, kv_scales[r * (d_nope / 128) + d / 128]));
          } else {
            row[d] = bf16_bits_to_double(((const uint16_t*)kv_nope)[r * d_nope + d]);
          }
        }
        for (int d = 0; d < d_rope; ++d) row[d_nope + d] = bf16_bits_to_double(kv_rope[r * d_rope + d]);
        ++nv;
      }
      for (int h = 0; h < n_q; ++h) {
        const int64_t qh = (int64_t)t * n_q + h;
        for (int d = 0; d < d_nope; ++d) q[d] = bf16_bits_to_double(q_nope[qh * d_nope + d]);
        for (int d = 0; d < d_rope; ++d) q[d_nope + d] = bf16_bits_to_double(q_rope[qh * d_rope + d]);
        double* o = out + ((int64_t)n * n_q + h) * d_nope;
        for (int d = 0; d < d_nope; ++d) o[d] = 0.0;
        if (nv == 0) {
          lse[(int64_t)n * n_q + h] = -INFINITY;
          continue;
        }
        /* step 3: scaled scores over the concatenated nope + rope dims */
        double m = -INFINITY;
        for (int i = 0; i < nv; ++i) {
          const double* row = K + (size_t)i * D;
          double s = 0.0;
          for (int d = 0; d < D; ++d) s += q[d] * row[d];
          z[i] = softmax_scale * s;
          if (z[i] > m) m = z[i];
        }
        /* steps 4-5: exact softmax, value = key_nope */
        double l = 0.0;
        for (int i = 0; i < nv; ++i) {
          const double p = exp(z[i] - m);
          l += p;
          const double* row = K + (size_t)i * D;
          for (int d = 0; d < d_nope; ++d) o[d] += p * row[d];
        }
        for (int d = 0; d < d_nope; ++d) o[d] /= l;
        lse[(int64_t)n * n_q + h] = m + log(l);
      }
    }
    free(K);
    free(z);
    free(q);
  }
  if (bad_blocks) *bad_blocks = bad_total;
  return 0;
}

int mla_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
