"""TEST INFRASTRUCTURE ONLY: the oracle for the MLA Prolog, which turns hidden
states into the attention's absorbed query and writes the new key row into
the paged cache.  Only tests/, the smoke check and the benchmark's
CPU-baseline leg may import it; the product path never does.

Written from "NPU DeepSeek-V4 PyPTO fused-operator optimization", section
MlaProlog (its two formula groups), shaped by the tensors of "CANN DeepSeek
Indexer attention" (section MLA Prolog: the V3 structure with weight
absorption in decode; the fused prototype's argument list x, w_dq, w_uq_qr,
w_uk, w_dkv_kr, gamma_cq, gamma_ckv, sin, cos, cache_index, kv_cache,
kr_cache) and by the cache of "DeepSeek V3/V2 Sparse Flash Attention with
Quantization" (512 latent + 64 rope, bf16 or INT8):

  query   c^Q = RMSNorm(x @ wq_a) * gamma_cq
          q   = RMSNorm(c^Q @ wq_b)            (per head, weight 1)
          q[..., -64:] = RoPE(q[..., -64:])   (interleaved)
          q_nope_abs[h] = q[h, :128] @ w_uk[h]  (absorption, 128 -> 512)
  key     k = RMSNorm(x @ wkv) * gamma_ckv     (the whole 576-wide row)
          k[-64:] = RoPE(k[-64:])
          the row k[:512] | k[512:] goes into the cache at cache_index.

Readings where the pages are open (kept identical in the CUDA path):
  - RMSNorm(v) = v / sqrt(mean(v^2) + eps) over the last axis; eps = 1e-6;
    the query's second RMSNorm runs per head over the head's 192 values
    (128 no-position + 64 rope), its weight fixed at 1;
  - the key's RMSNorm spans the whole x @ wkv row (512 + 64), as the formula
    normalises k before rotating its last rope_dim values;
  - interleaved RoPE pairs (2i, 2i + 1), i < 32, rotated by angle phi[t, i]
    given as cos[t, i], sin[t, i] (fp32 inputs, one angle per pair):
        y[2i]     = x[2i] cos - x[2i+1] sin
        y[2i + 1] = x[2i] sin + x[2i+1] cos
  - storage points: every tensor that a matrix product consumes (x, the
    weights, c^Q, q[:, :, :128]) and every cache row is bf16; between those
    points arithmetic is exact (fp64 here); gamma_cq and gamma_ckv are bf16;
  - the outputs q_nope_abs (T, H, 512) and q_rope (T, H, 64) are returned
    exact (fp64); the caller's bf16 copies round them;
  - the cache write follows the cache writer's rule (oracle.cache_write):
    negative cache_index skips the row, INT8 quantises the bf16 k row.
The fp64 steps use numpy; a matrix product is the only library step.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6
D_QK_NOPE = 128
D_ROPE = 64
D_LATENT = 512


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x):
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.  bf16 keeps
    8 significant bits: x = m * 2^e with m in [0.5, 1) rounds to
    rint(m * 2^8) * 2^(e - 8) (rint rounds halves to even)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def f64_to_bf16_bits(x):
    """Bits of round_bf16(x) (exact: a bf16 value is an fp32 value)."""
    v = round_bf16(x).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def rms_norm(v, gamma=None, eps=EPS):
    """v / sqrt(mean(v^2) + eps) over the last axis, times gamma if given."""
    v = np.asarray(v, dtype=np.float64)
    y = v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)
    return y if gamma is None else y * gamma


def rope_interleaved(v, cos, sin):
    """Rotate the pairs (v[..., 2i], v[..., 2i + 1]) by the angle whose cosine
    and sine are cos[..., i], sin[..., i] (broadcast over leading axes)."""
    v = np.asarray(v, dtype=np.float64)
    a, b = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * sin + b * cos
    return out


def forward(inp: dict, round_intermediates: bool = True, eps: float = EPS) -> dict:
    """The MLA Prolog on a workload dict (numpy; bf16 arrays as uint16 bits):
    x (T, hidden), wq_a (hidden, q_lora), gamma_cq (q_lora,), wq_b
    (q_lora, H * 192), w_uk (H, 128, 512), wkv (hidden, 576), gamma_ckv (576,),
    cos / sin (T, 32) fp32.

    Returns q_nope (T, H, 512) and q_rope (T, H, 64) fp64, k_nope (T, 512) and
    k_rope (T, 64) as bf16 bits (the cache rows), and the intermediates c_q
    (T, q_lora) and q_head (T, H, 192) for inspection.  With
    ``round_intermediates`` False every step is exact fp64 (the bf16 storage
    points are skipped), which the pins use to check the formulas alone."""
    rnd = round_bf16 if round_intermediates else (lambda a: a)
    x = bf16_to_f64(inp["x"])
    T = x.shape[0]
    H = int(inp["w_uk"].shape[0])
    cos = np.asarray(inp["cos"], dtype=np.float64)
    sin = np.asarray(inp["sin"], dtype=np.float64)
    # query: two projections with an RMSNorm after each
    c_q = rnd(rms_norm(x @ bf16_to_f64(inp["wq_a"]), bf16_to_f64(inp["gamma_cq"]), eps))
    q = (c_q @ bf16_to_f64(inp["wq_b"])).reshape(T, H, D_QK_NOPE + D_ROPE)
    q = rms_norm(q, None, eps)
    q_rope = rope_interleaved(q[..., D_QK_NOPE:], cos[:, None, :], sin[:, None, :])
    q_nope_n = rnd(q[..., :D_QK_NOPE])
    w_uk = bf16_to_f64(inp["w_uk"])                                  # (H, 128, 512)
    q_nope = np.matmul(q_nope_n.transpose(1, 0, 2), w_uk).transpose(1, 0, 2)   # head h: q[:, h] @ w_uk[h]
    # key: one projection, RMSNorm over the whole row, rope on its tail
    k = rms_norm(x @ bf16_to_f64(inp["wkv"]), bf16_to_f64(inp["gamma_ckv"]), eps)
    k_rope = rope_interleaved(k[:, D_LATENT:], cos, sin)
    k_nope_v = k[:, :D_LATENT]
    return dict(q_nope=q_nope, q_rope=q_rope, k_nope=f64_to_bf16_bits(k_nope_v), k_rope=f64_to_bf16_bits(k_rope),
                k_nope_exact=k_nope_v, k_rope_exact=k_rope, c_q=c_q,
                q_head=np.concatenate([q_nope_n, q_rope], axis=-1))


def forward_with_cache(inp: dict) -> tuple[dict, tuple]:
    """``forward`` plus the cache write of its key rows into copies of the
    workload's cache arrays.  Returns (forward's dict, (kv_nope, kv_rope,
    kv_scales, skipped_bad))."""
    from . import cache_write                                          # the cache writer's oracle

    out = forward(inp)
    cache = cache_write(out["k_nope"], out["k_rope"], inp["cache_index"], inp["kv_nope"], inp["kv_rope"],
                        inp.get("kv_scales"))
    return out, cache
