"""TEST INFRASTRUCTURE ONLY: the oracle for compressed and sparse compressed
flash attention (CFA / SCFA).  Only tests/, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.

Written from "NPU DeepSeek-V4 PyPTO fused-operator optimization":
  - section CFA: the KV cache has two sources, ori_kv (the original cache)
    taken under a sliding window, and cmp_kv (the Compressor's output) under
    causal attention;
  - section SCFA: as CFA, except that cmp_kv entries are picked by
    cmp_sparse_indices;
  - section Compressor: a compressed entry is produced when start_pos + 1 is a
    multiple of compress_ratio, so entry i summarises positions
    [i * r, (i + 1) * r).
Readings where the pages are open (kept identical in the CUDA path):
  - token (b, s) sits at position p = act_seqs[b] - S1 + s (its sequence's
    newest S1 positions are the query tokens);
  - ori part: positions [p - window + 1, p] that are >= 0;
  - compressed entry i is visible to the token iff (i + 1) * r - 1 <= p; CFA
    takes every visible entry, SCFA the entries of its cmp_sparse_indices row
    (negative or not visible: masked);
  - cmp_kv is laid out like the original cache (rows of 512 latent + 64 rope,
    bf16 or INT8 with four fp32 group scales) and paged through its own block
    table, 128 entries per block;
  - one softmax over the union of both parts (a multiset: an entry listed
    twice counts twice), the attention of "DeepSeek V3/V2 Sparse Flash
    Attention with Quantization" otherwise (INT8 -> fp32 times the group
    scale -> bf16, scores (q_nope . k_nope + q_rope . k_rope) * scale, value =
    k_nope);
  - block ids outside [0, num_blocks) mask the entry and are counted.
Plain numpy in fp64 after the bf16 / dequantised inputs; a matrix product is
the only library step.
"""
from __future__ import annotations

import numpy as np


def _bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f32_to_bf16_f64(x32):
    """fp32 -> bf16 (round to nearest, ties to even) -> fp64, for finite values."""
    u = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32)
    return (b << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _rows_latent(nope, scales, rows, int8):
    if not int8:
        return _bf16_f64(nope[rows])
    q = nope[rows].astype(np.float32)                                     # INT8 -> fp32, exact
    s = np.repeat(np.asarray(scales, np.float32)[rows], 128, axis=1)      # one scale per 128 elements
    return _f32_to_bf16_f64(q * s)                                        # one fp32 product, then bf16


def entries(inp, t, window, cmp_ratio, cmp_idx=None):
    """(source, logical index) pairs of token t: source 0 = ori position,
    source 1 = compressed entry; the visibility and window rules of the module
    docstring, before any block-table lookup."""
    S1 = inp["dims"]["S1"]
    b, s = divmod(t, S1)
    p = int(inp["act_seqs"][b]) - S1 + s
    out = [(0, j) for j in range(max(0, p - window + 1), p + 1)]
    if cmp_idx is None:
        cands = range(0, (p + 1) // cmp_ratio) if p >= 0 else range(0)
    else:
        cands = [int(i) for i in cmp_idx[t]]
    for i in cands:
        if i >= 0 and (i + 1) * cmp_ratio - 1 <= p:
            out.append((1, i))
    return out


def forward(inp, window: int, cmp_ratio: int, cmp_idx=None, tokens=None):
    """Returns (out fp64 (n, n_q, 512), lse fp64 (n, n_q), bad_entries)."""
    d = inp["dims"]
    S1, H = d["S1"], d["n_q"]
    int8 = bool(d["kv_int8"])
    T = d["B"] * S1
    toks = range(T) if tokens is None else tokens
    src = [(inp["kv_nope"], inp.get("kv_scales"), inp["kv_rope"], inp["block_table"], d["num_blocks"]),
           (inp["cmp_nope"], inp.get("cmp_scales"), inp["cmp_rope"], inp["cmp_block_table"], d["cmp_num_blocks"])]
    out = np.zeros((len(toks), H, 512))
    lse = np.full((len(toks), H), -np.inf)
    bad = 0
    for n, t in enumerate(toks):
        b = t // S1
        rows = [[], []]
        for sidx, j in entries(inp, t, window, cmp_ratio, cmp_idx):
            nope, scales, rope, bt, nb = src[sidx]
            slot = j // 128
            blk = int(bt[b, slot]) if slot < bt.shape[1] else -1
            if blk < 0 or blk >= nb:
                bad += 1
                continue
            rows[sidx].append(blk * 128 + j % 128)
        kn = [np.zeros((0, 512))]
        kr = [np.zeros((0, 64))]
        for sidx in (0, 1):
            if rows[sidx]:
                r = np.asarray(rows[sidx], dtype=np.int64)
                nope, scales, rope, _, _ = src[sidx]
                kn.append(_rows_latent(nope, scales, r, int8))
                kr.append(_bf16_f64(rope[r]))
        kn = np.concatenate(kn)
        kr = np.concatenate(kr)
        if kn.shape[0] == 0:
            continue
        qn, qr = _bf16_f64(inp["q_nope"][t]), _bf16_f64(inp["q_rope"][t])
        z = (qn @ kn.T + qr @ kr.T) * inp["softmax_scale"]
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        den = e.sum(axis=1)
        out[n] = (e @ kn) / den[:, None]
        lse[n] = m[:, 0] + np.log(den)
    return out, lse, bad
