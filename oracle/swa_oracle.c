/*
 * TEST INFRASTRUCTURE ONLY -- the oracle's window step for sliding-window
 * attention.  Only tests/, the smoke check and the benchmark's CPU-baseline
 * leg may load this library; the product path never calls it and shares no
 * code with it.
 *
 * "NPU DeepSeek-V4 PyPTO fused-operator optimization", section SWA: sliding
 * window attention over the original KV cache, the layer type used when the
 * compression ratio is 1, implemented by masking for prefill and MTP.  The
 * pages leave these points open; the readings used here:
 *   - the S1 query tokens of sequence b are its newest S1 positions:
 *     token (b, s) sits at position p = act_seqs[b] - S1 + s (the same
 *     convention as the decode / MTP and prefill workloads);
 *   - a token attends to the positions [p - window + 1, p] that are >= 0 (its
 *     own position included, nothing after it);
 *   - the window is a parameter (the pages give none).
 * The attention itself over those positions is the sparse attention
 * definition (mla_oracle.c), so this step only writes each token's position
 * list: entry e of token t is p - window + 1 + e, or -1 when that is negative.
 */
#include <stdint.h>

int swa_oracle_window_lists(int B, int S1, const int32_t* act_seqs, int window, int32_t* lists) {
  if (B <= 0 || S1 <= 0 || window <= 0) return -1;
  for (int b = 0; b < B; ++b) {
    for (int s = 0; s < S1; ++s) {
      const int64_t p = (int64_t)act_seqs[b] - S1 + s;
      int32_t* row = lists + ((int64_t)b * S1 + s) * window;
      for (int e = 0; e < window; ++e) {
        const int64_t j = p - window + 1 + e;
        row[e] = j >= 0 ? (int32_t)j : -1;
      }
    }
  }
  return 0;
}
