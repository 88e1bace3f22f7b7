/*
 * TEST INFRASTRUCTURE ONLY -- the oracle for the Lightning Indexer and its
 * top-k selection.  Only tests/, the smoke check and the benchmark's
 * CPU-baseline leg may load this library; the product path never calls it and
 * shares no code with it.
 *
 * Written from "CANN DeepSeek Indexer attention":
 *   - section "Lightning Indexer": the index score of query token i for cached
 *     key j is  I[i, j] = sum_h w[i, h] * ReLU(q[i, h, :] . k[j, :]),  with the
 *     head weights w[i, :] given per token (computed upstream);
 *   - section "Sparse Flash Attention": token i attends to the entries
 *     Top-k(I[i, :]).
 * The pages leave these points open; the readings used here:
 *   - the candidate keys of token t = (b, s) are the positions j in
 *     [0, act_seq[b]) of its sequence, paged exactly like the attention cache:
 *     row = block_table[b, j / block_size] * block_size + j % block_size; a
 *     position whose block id lies outside [0, num_blocks) (or whose table slot
 *     is beyond the table) is not a candidate and is counted as a bad block;
 *   - Top-k keeps the min(k, #candidates) largest scores; among equal scores
 *     the smaller position wins, which makes the selection unique;
 *   - the selected positions are returned in ascending order, padded with -1.
 *
 * Scores are exact: bf16 inputs widened to fp64, fp32 weights widened, fp64
 * arithmetic.  The selection works on any array of scores (fp64 here), so the
 * same rule can be applied to scores computed in another precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double idx_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * scores: (B*S1, ld) fp64; entry [t, j] is I[t, j] for candidate positions and
 * -inf otherwise (including j >= act_seq[b]).  ld >= max_blocks_per_seq *
 * block_size.  Returns 0, or a negative value on bad arguments.
 */
int idx_oracle_scores(int B, int S1, int H, int D, int block_size, int num_blocks, int max_blocks_per_seq,
                      const uint16_t* q, const float* w, const uint16_t* k_cache, const int32_t* block_table,
                      const int32_t* act_seqs, int ld, double* scores, int n_threads, int64_t* bad_blocks) {
  if (B <= 0 || S1 <= 0 || H <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
      ld < max_blocks_per_seq * block_size)
    return -1;
  const int T = B * S1;
  int64_t bad_total = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 1) reduction(+ : bad_total)
#endif
  for (int t = 0; t < T; ++t) {
    const int b = t / S1;
    const int act = act_seqs[b];
    double* row_out = scores + (int64_t)t * ld;
    for (int j = 0; j < ld; ++j) row_out[j] = -INFINITY;
    for (int j = 0; j < act && j < ld; ++j) {
      const int slot = j / block_size;
      const int blk = slot < max_blocks_per_seq ? block_table[(int64_t)b * max_blocks_per_seq + slot] : -1;
      if (blk < 0 || blk >= num_blocks) {
        ++bad_total;
        continue;
      }
      const uint16_t* kr = k_cache + ((int64_t)blk * block_size + j % block_size) * D;
      double acc = 0.0;
      for (int h = 0; h < H; ++h) {
        const uint16_t* qr = q + ((int64_t)t * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += idx_bf16(qr[d]) * idx_bf16(kr[d]);
        acc += (double)w[(int64_t)t * H + h] * (dot > 0.0 ? dot : 0.0);
      }
      row_out[j] = acc;
    }
  }
  if (bad_blocks) *bad_blocks = bad_total;
  return 0;
}

typedef struct {
  double s;
  int32_t j;
} idx_entry;

/* larger score first; equal scores: smaller position first */
static int idx_by_score(const void* a, const void* b) {
  const idx_entry* x = (const idx_entry*)a;
  const idx_entry* y = (const idx_entry*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

static int idx_by_pos(const void* a, const void* b) {
  const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/*
 * Top-k over scores[t, 0:act_seq[b]) (fp64, -inf marks a non-candidate):
 * out (B*S1, topk) int32, ascending positions, -1 padded.  Returns 0.
 */
int idx_oracle_select(int B, int S1, const int32_t* act_seqs, int ld, const double* scores, int topk, int32_t* out) {
  if (B <= 0 || S1 <= 0 || topk <= 0 || ld <= 0) return -1;
  const int T = B * S1;
  idx_entry* e = (idx_entry*)malloc(sizeof(idx_entry) * (size_t)ld);
  int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)topk);
  for (int t = 0; t < T; ++t) {
    const int act = act_seqs[t / S1] < ld ? act_seqs[t / S1] : ld;
    int n = 0;
    for (int j = 0; j < act; ++j) {
      const double s = scores[(int64_t)t * ld + j];
      if (s == -INFINITY) continue; /* not a candidate */
      e[n].s = s;
      e[n].j = j;
      ++n;
    }
    qsort(e, (size_t)n, sizeof(idx_entry), idx_by_score);
    const int m = n < topk ? n : topk;
    for (int i = 0; i < m; ++i) sel[i] = e[i].j;
    qsort(sel, (size_t)m, sizeof(int32_t), idx_by_pos);
    for (int i = 0; i < topk; ++i) out[(int64_t)t * topk + i] = i < m ? sel[i] : -1;
  }
  free(e);
  free(sel);
  return 0;
}
