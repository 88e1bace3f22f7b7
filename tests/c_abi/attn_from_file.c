/*
 * A plain C caller of the library's C ABI (no Python, no torch): reads one
 * attention problem from a binary file, runs mla_sparse_attn_fwd on the
 * default stream and writes out (bf16) and lse (fp32) to another file.
 *
 * Input file: 11 int32 (B, S1, n_q, num_blocks, max_blocks_per_seq, topk,
 * kv_int8, mode, then three zeros), one float32 softmax_scale, then the
 * arrays in this order with the sizes of include/mla_sparse.h: q_nope,
 * q_rope, kv_nope, kv_rope, kv_scales (INT8 only), topk_idx, block_table,
 * act_seqs.  Output file: out then lse.  Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "mla_sparse.h"

static void* read_block(FILE* f, size_t bytes) {
  void* h = malloc(bytes ? bytes : 1);
  if (!h || fread(h, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read (%zu bytes)\n", bytes);
    exit(2);
  }
  return h;
}

static void* to_device(const void* h, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "device copy failed\n");
    exit(3);
  }
  return d;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input.bin output.bin\n", argv[0]);
    return 1;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 1;
  int32_t hdr[11];
  float scale;
  if (fread(hdr, sizeof hdr, 1, f) != 1 || fread(&scale, sizeof scale, 1, f) != 1) return 2;
  mla_dims d;
  d.B = hdr[0];
  d.S1 = hdr[1];
  d.n_q = hdr[2];
  d.n_kv = 1;
  d.d_nope = 512;
  d.d_rope = 64;
  d.block_size = 128;
  d.num_blocks = hdr[3];
  d.max_blocks_per_seq = hdr[4];
  d.topk = hdr[5];
  d.kv_dtype = hdr[6] ? MLA_KV_INT8 : MLA_KV_BF16;
  const int32_t mode = hdr[7];
  const size_t T = (size_t)d.B * d.S1, rows = (size_t)d.num_blocks * 128;
  const size_t b_qn = T * d.n_q * 512 * 2, b_qr = T * d.n_q * 64 * 2;
  const size_t b_kn = rows * 512 * (d.kv_dtype == MLA_KV_INT8 ? 1 : 2), b_kr = rows * 64 * 2;
  const size_t b_ks = d.kv_dtype == MLA_KV_INT8 ? rows * 4 * 4 : 0;
  const size_t b_tk = T * d.topk * 4, b_bt = (size_t)d.B * d.max_blocks_per_seq * 4, b_as = (size_t)d.B * 4;
  void* h_qn = read_block(f, b_qn);
  void* h_qr = read_block(f, b_qr);
  void* h_kn = read_block(f, b_kn);
  void* h_kr = read_block(f, b_kr);
  void* h_ks = b_ks ? read_block(f, b_ks) : NULL;
  void* h_tk = read_block(f, b_tk);
  void* h_bt = read_block(f, b_bt);
  void* h_as = read_block(f, b_as);
  fclose(f);
  void* qn = to_device(h_qn, b_qn);
  void* qr = to_device(h_qr, b_qr);
  void* kn = to_device(h_kn, b_kn);
  void* kr = to_device(h_kr, b_kr);
  float* ks = b_ks ? (float*)to_device(h_ks, b_ks) : NULL;
  int32_t* tk = (int32_t*)to_device(h_tk, b_tk);
  int32_t* bt = (int32_t*)to_device(h_bt, b_bt);
  int32_t* as = (int32_t*)to_device(h_as, b_as);
  const size_t b_out = T * d.n_q * 512 * 2, b_lse = T * d.n_q * 4;
  void* out = NULL;
  float* lse = NULL;
  if (cudaMalloc(&out, b_out) != cudaSuccess || cudaMalloc((void**)&lse, b_lse) != cudaSuccess) return 3;
  const mla_status st = mla_sparse_attn_fwd(&d, qn, qr, kn, kr, ks, tk, bt, as, out, lse, scale, mode, NULL);
  if (st != MLA_OK) {
    fprintf(stderr, "mla_sparse_attn_fwd: %d %s\n", (int)st, mla_sparse_last_error());
    return 4;
  }
  uint32_t flags = 0;
  if (mla_sparse_device_status(NULL, &flags, 1) != MLA_OK) {
    fprintf(stderr, "device status 0x%x: %s\n", flags, mla_sparse_last_error());
    return 5;
  }
  void* h_out = malloc(b_out);
  void* h_lse = malloc(b_lse);
  if (cudaMemcpy(h_out, out, b_out, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(h_lse, lse, b_lse, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 3;
  FILE* o = fopen(argv[2], "wb");
  if (!o || fwrite(h_out, 1, b_out, o) != b_out || fwrite(h_lse, 1, b_lse, o) != b_lse) return 6;
  fclose(o);
  return 0;
}
