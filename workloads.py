"""Seeded synthetic inputs for sparse MLA attention over a paged KV cache.

This module only draws inputs; it contains none of the attention arithmetic.
Both the oracle (``oracle/``) and the CUDA path receive exactly the arrays
built here, generated on the CPU with ``torch.Generator().manual_seed(seed)``
and handed over as numpy arrays (bf16 values as their uint16 bit patterns).

Layouts (row-major, the operator's I/O table):
  q_nope  (B*S1, n_q, 512) bf16      q_rope (B*S1, n_q, 64) bf16
  kv_nope (num_blocks*128, 512) bf16 | int8
  kv_rope (num_blocks*128, 64) bf16  kv_scales (num_blocks*128, 4) fp32 (INT8 only)
  topk_idx (B*S1, topk) int32        block_table (B, max_blocks_per_seq) int32
  act_seqs (B,) int32

The five named workloads follow the shapes of the pages' test cases and timing
table (B=64, S1=2, S2=8192, D=512; act_seq up to 65536; a prefill run) with
q/k drawn from N(0, 1).  No public dataset is involved.
"""
from __future__ import annotations

import math

import numpy as np
import torch

D_NOPE = 512
D_ROPE = 64
BLOCK_SIZE = 128
BF16_NAN_BITS = 0x7FC0


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _randn_bf16(g: torch.Generator, shape, chunk_rows: int = 1 << 16) -> np.ndarray:
    """N(0, 1) rounded to bf16, drawn in row chunks to bound peak memory."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = _bf16_bits(torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g))
    return out


def quantize_int8_groups(x: torch.Tensor):
    """Per-row INT8 with one fp32 scale per 128-element group.

    scale = absmax / 127 (a group of zeros gets scale 1), q = clamp(round(x / scale),
    -128, 127) with round-half-to-even.  This is how the synthetic INT8 cache is
    written; the attention path only ever reads q and scale back.
    """
    rows, d = x.shape
    grp = x.reshape(rows, d // 128, 128)
    absmax = grp.abs().amax(dim=-1)
    scale = absmax / 127.0
    scale = torch.where(absmax > 0, scale, torch.ones_like(scale))
    q = torch.round(grp / scale[..., None]).clamp_(-128, 127).to(torch.int8)
    return q.reshape(rows, d).numpy(), scale.to(torch.float32).numpy()


def make_inputs(*, B: int, S1: int, n_q: int, act_seqs, topk: int, seed: int, num_blocks: int | None = None,
                max_blocks_per_seq: int | None = None, kv_int8: bool = False, positions=None,
                poison_unused: bool = True, softmax_scale: float | None = None, mode: str = "decode",
                name: str = "custom") -> dict:
    """Build one workload.

    act_seqs: per-batch actual KV length.  Each batch gets ceil(act/128)
    physical blocks, drawn without replacement from a random permutation of
    ``num_blocks`` (default: exactly the blocks needed); the table is padded
    with -1.  ``positions`` (optional, (B, S1)) gives each token's position p:
    the token then selects among [0, p] (causal prefill); otherwise among
    [0, act).  A token selects min(topk, n) distinct indices uniformly (n =
    its candidate count) in random order, padded with -1.  Cache rows that no
    valid index can reach (unused blocks, positions >= act) are NaN when
    ``poison_unused``.
    """
    g = torch.Generator().manual_seed(int(seed))
    act = np.asarray(act_seqs, dtype=np.int64).reshape(B)
    nb = [(int(a) + BLOCK_SIZE - 1) // BLOCK_SIZE for a in act]
    used = int(sum(nb))
    if num_blocks is None:
        num_blocks = max(used, 1)
    if num_blocks < used:
        raise ValueError("num_blocks smaller than the blocks the sequences need")
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(max(nb), 1)
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    block_table = np.full((B, max_blocks_per_seq), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        block_table[b, : nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    T = B * S1
    topk_idx = np.full((T, topk), -1, dtype=np.int32)
    for t in range(T):
        b = t // S1
        n_cand = int(act[b]) if positions is None else int(np.asarray(positions)[b, t % S1]) + 1
        n_cand = max(0, min(n_cand, int(act[b])))
        k = min(topk, n_cand)
        if k > 0:
            topk_idx[t, :k] = torch.randperm(n_cand, generator=g)[:k].numpy().astype(np.int32)
    rows = num_blocks * BLOCK_SIZE
    if kv_int8:
        kv_nope = np.empty((rows, D_NOPE), dtype=np.int8)
        kv_scales = np.empty((rows, D_NOPE // 128), dtype=np.float32)
        step = 1 << 15
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            q8, sc = quantize_int8_groups(torch.randn((r1 - r0, D_NOPE), generator=g))
            kv_nope[r0:r1] = q8
            kv_scales[r0:r1] = sc
    else:
        kv_nope = _randn_bf16(g, (rows, D_NOPE))
        kv_scales = None
    kv_rope = _randn_bf16(g, (rows, D_ROPE))
    q_nope = _randn_bf16(g, (T, n_q, D_NOPE))
    q_rope = _randn_bf16(g, (T, n_q, D_ROPE))
    if poison_unused:
        reach = np.zeros(rows, dtype=bool)
        for b in range(B):
            for s in range(nb[b]):
                blk = block_table[b, s]
                lo = blk * BLOCK_SIZE
                n_valid = min(BLOCK_SIZE, int(act[b]) - s * BLOCK_SIZE)
                reach[lo:lo + n_valid] = True
        dead = ~reach
        if dead.any():
            kv_rope[dead] = BF16_NAN_BITS
            if kv_int8:
                kv_scales[dead] = np.nan
            else:
                kv_nope[dead] = BF16_NAN_BITS
    dims = dict(B=B, S1=S1, n_q=n_q, n_kv=1, d_nope=D_NOPE, d_rope=D_ROPE, block_size=BLOCK_SIZE,
                num_blocks=int(num_blocks), max_blocks_per_seq=int(max_blocks_per_seq), topk=int(topk),
                kv_int8=int(bool(kv_int8)))
    return dict(name=name, dims=dims, q_nope=q_nope, q_rope=q_rope, kv_nope=kv_nope, kv_rope=kv_rope,
                kv_scales=kv_scales, topk_idx=topk_idx, block_table=block_table,
                act_seqs=act.astype(np.int32),
                softmax_scale=float(softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(D_NOPE + D_ROPE)),
                mode=mode)


# ------------------------------------------------------------------ named workloads
def tiny_decode(seed: int = 0) -> dict:
    """B=1 S1=1 H=16, act 256 over 2 of 4 physical blocks (2 NaN-filled), topk 64."""
    return make_inputs(B=1, S1=1, n_q=16, act_seqs=[256], topk=64, num_blocks=4, seed=seed, name="tiny_decode")


def mtp_decode(seed: int = 1, B: int = 64) -> dict:
    """B=64 S1=2 H=128, act 8192 each, 4096 shuffled blocks, topk 2048 distinct, bf16."""
    return make_inputs(B=B, S1=2, n_q=128, act_seqs=[8192] * B, topk=2048, seed=seed, name="mtp_decode")


def mtp_decode_b2(seed: int = 16) -> dict:
    """Low-batch MTP decode: B=2 S1=2 (4 query tokens), otherwise as mtp_decode."""
    return make_inputs(B=2, S1=2, n_q=128, act_seqs=[8192] * 2, topk=2048, seed=seed, name="mtp_decode_b2")


def int8_decode(seed: int = 2, B: int = 64) -> dict:
    """As mtp_decode with key_nope INT8 per 128-group (scale = absmax/127)."""
    return make_inputs(B=B, S1=2, n_q=128, act_seqs=[8192] * B, topk=2048, seed=seed, kv_int8=True,
                       name="int8_decode")


def varlen_decode(seed: int = 3, B: int = 64) -> dict:
    """B=64 S1=2 H=128 topk 2048, act_b ~ U{512..65536}, shuffled blocks, -1 padding."""
    g = torch.Generator().manual_seed(int(seed) + 1000)
    act = torch.randint(512, 65537, (B,), generator=g).numpy()
    return make_inputs(B=B, S1=2, n_q=128, act_seqs=act, topk=2048, seed=seed, name="varlen_decode")


def swa_decode(seed: int = 10, B: int = 64, window: int = 128) -> dict:
    """Sliding-window attention inputs: B=64 S1=2 H=128, act 8192 each, 4096
    shuffled blocks, bf16; the window is a parameter (the pages give none).
    The top-k list that make_inputs draws is not used by this workload."""
    inp = make_inputs(B=B, S1=2, n_q=128, act_seqs=[8192] * B, topk=64, seed=seed, name="swa_decode")
    inp["window"] = int(window)
    return inp


def prefill(seed: int = 4, B: int = 4, S1: int = 1024) -> dict:
    """B=4, S1=1024 tokens at positions 7168..8191 of act 8192, causal top-2048."""
    act = 8192
    pos = np.tile(np.arange(act - S1, act, dtype=np.int64), (B, 1))
    return make_inputs(B=B, S1=S1, n_q=128, act_seqs=[act] * B, topk=2048, seed=seed, positions=pos,
                       mode="prefill", name="prefill")


NAMED = {
    "tiny_decode": tiny_decode,
    "mtp_decode": mtp_decode,
    "mtp_decode_b2": mtp_decode_b2,
    "int8_decode": int8_decode,
    "varlen_decode": varlen_decode,
    "prefill": prefill,
    "swa_decode": swa_decode,
}


def to_device(inp: dict, device="cuda") -> dict:
    """Copy a workload to the device as torch tensors, plus empty out / lse."""
    d = inp["dims"]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def raw(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    dev = dict(q_nope=bf(inp["q_nope"]), q_rope=bf(inp["q_rope"]),
               kv_nope=raw(inp["kv_nope"]) if d["kv_int8"] else bf(inp["kv_nope"]), kv_rope=bf(inp["kv_rope"]),
               kv_scales=raw(inp["kv_scales"]) if d["kv_int8"] else None, topk_idx=raw(inp["topk_idx"]),
               block_table=raw(inp["block_table"]), act_seqs=raw(inp["act_seqs"]))
    T, H = d["B"] * d["S1"], d["n_q"]
    dev["out"] = torch.empty((T, H, d["d_nope"]), dtype=torch.bfloat16, device=device)
    dev["lse"] = torch.empty((T, H), dtype=torch.float32, device=device)
    return dev


# ------------------------------------------------------------------ Lightning Indexer inputs
INDEXER_HEADS = 64
INDEXER_DIM = 128


def make_indexer_inputs(*, B: int, S1: int, act_seqs, topk: int, seed: int, n_heads: int = INDEXER_HEADS,
                        head_dim: int = INDEXER_DIM, num_blocks: int | None = None,
                        max_blocks_per_seq: int | None = None, poison_unused: bool = True,
                        w_scale: float = 1.0, name: str = "custom") -> dict:
    """One Lightning Indexer workload: q (B*S1, H, D) bf16 ~ N(0, 1), the
    per-token head weights w (B*S1, H) fp32 ~ N(0, w_scale^2), and a paged
    index-key cache k_cache (num_blocks*128, D) bf16 ~ N(0, 1) with the same
    block-table construction as make_inputs (rows no candidate can reach are
    NaN when ``poison_unused``)."""
    g = torch.Generator().manual_seed(int(seed))
    act = np.asarray(act_seqs, dtype=np.int64).reshape(B)
    nb = [(int(a) + BLOCK_SIZE - 1) // BLOCK_SIZE for a in act]
    used = int(sum(nb))
    if num_blocks is None:
        num_blocks = max(used, 1)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(max(nb), 1)
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    block_table = np.full((B, max_blocks_per_seq), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        block_table[b, : nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    T = B * S1
    k_cache = _randn_bf16(g, (num_blocks * BLOCK_SIZE, head_dim))
    q = _randn_bf16(g, (T, n_heads, head_dim))
    w = (torch.randn((T, n_heads), generator=g) * w_scale).to(torch.float32).numpy()
    if poison_unused:
        reach = np.zeros(num_blocks * BLOCK_SIZE, dtype=bool)
        for b in range(B):
            for s in range(nb[b]):
                lo = block_table[b, s] * BLOCK_SIZE
                reach[lo:lo + min(BLOCK_SIZE, int(act[b]) - s * BLOCK_SIZE)] = True
        k_cache[~reach] = BF16_NAN_BITS
    dims = dict(B=B, S1=S1, n_heads=n_heads, head_dim=head_dim, block_size=BLOCK_SIZE, num_blocks=int(num_blocks),
                max_blocks_per_seq=int(max_blocks_per_seq), topk=int(topk))
    return dict(name=name, dims=dims, q=q, w=w, k_cache=k_cache, block_table=block_table,
                act_seqs=act.astype(np.int32))


def indexer_decode(seed: int = 5, B: int = 64) -> dict:
    """B=64 S1=2, 64 heads x 128 dims, act 8192 each over 4096 shuffled blocks, top-2048."""
    return make_indexer_inputs(B=B, S1=2, act_seqs=[8192] * B, topk=2048, seed=seed, name="indexer_decode")


def indexer_tiny(seed: int = 6) -> dict:
    """B=1 S1=1, 16 heads, act 300 (3 of 5 blocks, the last partial), top-64."""
    return make_indexer_inputs(B=1, S1=1, n_heads=16, act_seqs=[300], topk=64, num_blocks=5, seed=seed,
                               name="indexer_tiny")


def indexer_varlen(seed: int = 7, B: int = 8) -> dict:
    """B=8 S1=2, act_b ~ U{100..20000} (some below top-k), top-2048."""
    g = torch.Generator().manual_seed(int(seed) + 1000)
    act = torch.randint(100, 20001, (B,), generator=g).numpy()
    return make_indexer_inputs(B=B, S1=2, act_seqs=act, topk=2048, seed=seed, name="indexer_varlen")


INDEXER_NAMED = {
    "indexer_tiny": indexer_tiny,
    "indexer_decode": indexer_decode,
    "indexer_varlen": indexer_varlen,
}


def indexer_to_device(inp: dict, device="cuda") -> dict:
    """Copy an indexer workload to the device, plus empty topk / scores outputs."""
    d = inp["dims"]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def raw(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    T = d["B"] * d["S1"]
    dev = dict(q=bf(inp["q"]), w=raw(inp["w"]), k_cache=bf(inp["k_cache"]), block_table=raw(inp["block_table"]),
               act_seqs=raw(inp["act_seqs"]))
    dev["topk_idx"] = torch.empty((T, d["topk"]), dtype=torch.int32, device=device)
    dev["scores"] = torch.empty((T, d["max_blocks_per_seq"] * d["block_size"]), dtype=torch.float32, device=device)
    return dev


# ------------------------------------------------------------------ paged cache writer
def make_cache_write_inputs(*, T: int, num_blocks: int, kv_int8: bool, seed: int, skip_every: int = 17,
                            name: str = "custom") -> dict:
    """New key rows for the paged cache writer and the cache they go into.

    k_nope (T, 512) bf16 ~ N(0, s_t^2) with a per-row s_t ~ U(0.01, 10), plus
    special rows (a zero group, exact multiples of 2^-3 with a +-127 extreme,
    half-way ties at scale 1); k_rope (T, 64) bf16 ~ N(0, 1); cache_index:
    distinct random flat rows, every ``skip_every``-th entry -1.  The existing
    cache holds random rows (bf16, or INT8 codes with scales)."""
    g = torch.Generator().manual_seed(int(seed))
    rows = num_blocks * BLOCK_SIZE
    assert T <= rows
    scale_t = torch.empty((T, 1)).uniform_(0.01, 10.0, generator=g)
    x = torch.randn((T, D_NOPE), generator=g) * scale_t
    if T >= 3:
        x[0, 128:256] = 0.0
        k = torch.randint(-127, 128, (D_NOPE,), generator=g).to(torch.float32)
        k[5] = 127.0
        k[133] = -127.0
        k[261] = 127.0
        k[389] = -127.0
        x[1] = k * 2.0 ** -3
        x[2] = 0.0
        x[2, 0] = 127.0
        x[2, 1:9] = torch.tensor([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5])
    k_nope = _bf16_bits(x)
    k_rope = _bf16_bits(torch.randn((T, D_ROPE), generator=g))
    idx = torch.randperm(rows, generator=g)[:T].to(torch.int64).numpy()
    if skip_every:
        idx[::skip_every] = -1
    kv_rope = _bf16_bits(torch.randn((rows, D_ROPE), generator=g))
    if kv_int8:
        kv_nope = torch.randint(-127, 128, (rows, D_NOPE), generator=g).to(torch.int8).numpy()
        kv_scales = torch.empty((rows, 4)).uniform_(0.001, 0.1, generator=g).numpy().astype(np.float32)
    else:
        kv_nope = _bf16_bits(torch.randn((rows, D_NOPE), generator=g))
        kv_scales = None
    return dict(name=name, k_nope=k_nope, k_rope=k_rope, cache_index=idx, kv_nope=kv_nope, kv_rope=kv_rope,
                kv_scales=kv_scales, dims=dict(T=T, num_blocks=num_blocks, kv_int8=int(bool(kv_int8))))


def cache_write_decode(seed: int = 8) -> dict:
    """128 new rows (B=64 x S1=2 decode tokens) into an INT8 cache of 4096 blocks."""
    return make_cache_write_inputs(T=128, num_blocks=4096, kv_int8=True, seed=seed, skip_every=0,
                                   name="cache_write_decode")


def cache_write_prefill(seed: int = 9) -> dict:
    """4096 new rows (B=4 x 1024 prefill tokens) into an INT8 cache of 4096 blocks."""
    return make_cache_write_inputs(T=4096, num_blocks=4096, kv_int8=True, seed=seed, skip_every=0,
                                   name="cache_write_prefill")


CACHE_WRITE_NAMED = {
    "cache_write_decode": cache_write_decode,
    "cache_write_prefill": cache_write_prefill,
}


def cache_write_to_device(inp: dict, device="cuda") -> dict:
    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def raw(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    int8 = inp["dims"]["kv_int8"]
    return dict(k_nope=bf(inp["k_nope"]), k_rope=bf(inp["k_rope"]), cache_index=raw(inp["cache_index"]),
                kv_nope=raw(inp["kv_nope"]) if int8 else bf(inp["kv_nope"]), kv_rope=bf(inp["kv_rope"]),
                kv_scales=raw(inp["kv_scales"]) if int8 else None)


# ------------------------------------------------------------------ compressed attention (CFA / SCFA)
def make_compressed_inputs(*, B: int, S1: int, n_q: int, act_seqs, window: int, cmp_ratio: int, seed: int,
                           cmp_topk: int | None = None, kv_int8: bool = False, name: str = "custom") -> dict:
    """Original cache and query as make_inputs, plus a compressed cache: entry i
    of sequence b exists for (i + 1) * cmp_ratio <= act_b, rows ~ N(0, 1) (bf16,
    or INT8 with group scales), paged through its own shuffled block table.
    With ``cmp_topk`` (SCFA) each token gets a list of cmp_topk distinct
    compressed entries drawn from its visible ones (padded with -1); without
    it (CFA) there is no list."""
    base = make_inputs(B=B, S1=S1, n_q=n_q, act_seqs=act_seqs, topk=1, seed=seed, kv_int8=kv_int8, name=name)
    g = torch.Generator().manual_seed(int(seed) + 77)
    act = np.asarray(base["act_seqs"], dtype=np.int64)
    n_cmp = act // cmp_ratio
    nb = [max(1, (int(c) + BLOCK_SIZE - 1) // BLOCK_SIZE) for c in n_cmp]
    cnb = int(sum(nb))
    perm = torch.randperm(cnb, generator=g).numpy().astype(np.int32)
    cbt = np.full((B, max(nb)), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        cbt[b, : nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    rows = cnb * BLOCK_SIZE
    cmp_rope = _randn_bf16(g, (rows, D_ROPE))
    if kv_int8:
        q8, sc = quantize_int8_groups(torch.randn((rows, D_NOPE), generator=g))
        cmp_nope, cmp_scales = q8, sc
    else:
        cmp_nope, cmp_scales = _randn_bf16(g, (rows, D_NOPE)), None
    out = dict(base, cmp_nope=cmp_nope, cmp_rope=cmp_rope, cmp_scales=cmp_scales, cmp_block_table=cbt)
    out["dims"] = dict(base["dims"], cmp_num_blocks=cnb, cmp_max_blocks_per_seq=int(cbt.shape[1]),
                       window=int(window), cmp_ratio=int(cmp_ratio), cmp_topk=int(cmp_topk or 0))
    if cmp_topk:
        T = B * S1
        lists = np.full((T, cmp_topk), -1, dtype=np.int32)
        for t in range(T):
            b, s = divmod(t, S1)
            p = int(act[b]) - S1 + s
            vis = max(0, (p + 1) // cmp_ratio)
            k = min(cmp_topk, vis)
            if k:
                lists[t, :k] = torch.randperm(vis, generator=g)[:k].numpy()
        out["cmp_idx"] = lists
    return out


def cfa_decode(seed: int = 11, B: int = 64) -> dict:
    """CFA: B=64 S1=2 H=128, act 8192, window 128, compression ratio 128 (64 compressed entries)."""
    return make_compressed_inputs(B=B, S1=2, n_q=128, act_seqs=[8192] * B, window=128, cmp_ratio=128, seed=seed,
                                  name="cfa_decode")


def scfa_decode(seed: int = 12, B: int = 64) -> dict:
    """SCFA: B=64 S1=2 H=128, act 8192, window 128, ratio 4 (2048 compressed entries), 512 selected per token."""
    return make_compressed_inputs(B=B, S1=2, n_q=128, act_seqs=[8192] * B, window=128, cmp_ratio=4, cmp_topk=512,
                                  seed=seed, name="scfa_decode")


COMPRESSED_NAMED = {"cfa_decode": cfa_decode, "scfa_decode": scfa_decode}


# ------------------------------------------------------------------ MLA Prolog (synthetic weights)
PROLOG_HIDDEN = 7168
PROLOG_Q_LORA = 1536
PROLOG_HEADS = 128
PROLOG_QK_NOPE = 128
PROLOG_KV = D_NOPE + D_ROPE


def _randn_bf16_scaled(g: torch.Generator, shape, std: float, chunk_rows: int = 1 << 12) -> np.ndarray:
    """N(0, std^2) rounded to bf16, drawn in row chunks."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = _bf16_bits(torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g) * std)
    return out


def make_prolog_inputs(*, T: int, seed: int, hidden: int = PROLOG_HIDDEN, q_lora: int = PROLOG_Q_LORA,
                       n_heads: int = PROLOG_HEADS, num_blocks: int = 4096, kv_int8: bool = True,
                       skip_every: int = 0, name: str = "custom") -> dict:
    """Hidden states, random-init weights and a paged cache for the MLA Prolog.

    x (T, hidden) bf16 ~ N(0, 1), row 1 all zeros and row 2 scaled by 2^10 when
    T >= 3; weights bf16 ~ N(0, 1/fan_in): wq_a (hidden, q_lora), wq_b
    (q_lora, H*192), w_uk (H, 128, 512), wkv (hidden, 576); gamma_cq (q_lora,)
    and gamma_ckv (576,) bf16 ~ U(0.5, 1.5); cos / sin (T, 32) fp32 of angles
    ~ U(0, 2 pi); cache_index: distinct random flat rows (every
    ``skip_every``-th -1); the existing cache holds random rows (bf16, or INT8
    codes with scales).  No trained weights are involved."""
    g = torch.Generator().manual_seed(int(seed))
    H = int(n_heads)
    xs = torch.randn((T, hidden), generator=g)
    if T >= 3:
        xs[1] = 0.0
        xs[2] *= 2.0 ** 10
    x = _bf16_bits(xs)
    wq_a = _randn_bf16_scaled(g, (hidden, q_lora), hidden ** -0.5)
    wq_b = _randn_bf16_scaled(g, (q_lora, H * (PROLOG_QK_NOPE + D_ROPE)), q_lora ** -0.5)
    w_uk = _randn_bf16_scaled(g, (H, PROLOG_QK_NOPE, D_NOPE), PROLOG_QK_NOPE ** -0.5)
    wkv = _randn_bf16_scaled(g, (hidden, PROLOG_KV), hidden ** -0.5)
    gamma_cq = _bf16_bits(torch.empty(q_lora).uniform_(0.5, 1.5, generator=g))
    gamma_ckv = _bf16_bits(torch.empty(PROLOG_KV).uniform_(0.5, 1.5, generator=g))
    phi = torch.empty((T, D_ROPE // 2)).uniform_(0.0, 2.0 * math.pi, generator=g)
    cos = torch.cos(phi).numpy().astype(np.float32)
    sin = torch.sin(phi).numpy().astype(np.float32)
    rows = num_blocks * BLOCK_SIZE
    assert T <= rows
    idx = torch.randperm(rows, generator=g)[:T].to(torch.int64).numpy()
    if skip_every:
        idx[::skip_every] = -1
    kv_rope = _randn_bf16(g, (rows, D_ROPE))
    if kv_int8:
        kv_nope = torch.randint(-127, 128, (rows, D_NOPE), generator=g).to(torch.int8).numpy()
        kv_scales = torch.empty((rows, 4)).uniform_(0.001, 0.1, generator=g).numpy().astype(np.float32)
    else:
        kv_nope = _randn_bf16(g, (rows, D_NOPE))
        kv_scales = None
    return dict(name=name, x=x, wq_a=wq_a, gamma_cq=gamma_cq, wq_b=wq_b, w_uk=w_uk, wkv=wkv, gamma_ckv=gamma_ckv,
                cos=cos, sin=sin, cache_index=idx, kv_nope=kv_nope, kv_rope=kv_rope, kv_scales=kv_scales,
                dims=dict(T=T, hidden=hidden, q_lora=q_lora, n_heads=H, num_blocks=num_blocks,
                          kv_int8=int(bool(kv_int8))))


def prolog_tiny(seed: int = 13) -> dict:
    """13 tokens, hidden 256, q_lora 128, 4 heads, bf16 cache of 4 blocks, every 5th row skipped."""
    return make_prolog_inputs(T=13, seed=seed, hidden=256, q_lora=128, n_heads=4, num_blocks=4, kv_int8=False,
                              skip_every=5, name="prolog_tiny")


def prolog_decode(seed: int = 14) -> dict:
    """128 tokens (B=64 x S1=2 decode), DeepSeek-V3.2 sizes (hidden 7168, q_lora 1536, 128 heads),
    INT8 cache of 4096 blocks."""
    return make_prolog_inputs(T=128, seed=seed, num_blocks=4096, kv_int8=True, name="prolog_decode")


def prolog_prefill(seed: int = 15) -> dict:
    """1000 tokens (a ragged prefill chunk), DeepSeek-V3.2 sizes, bf16 cache of 4096 blocks."""
    return make_prolog_inputs(T=1000, seed=seed, num_blocks=4096, kv_int8=False, name="prolog_prefill")


PROLOG_NAMED = {"prolog_decode": prolog_decode, "prolog_prefill": prolog_prefill}


def prolog_to_device(inp: dict, device="cuda") -> dict:
    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def raw(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    int8 = inp["dims"]["kv_int8"]
    out = {k: bf(inp[k]) for k in ("x", "wq_a", "gamma_cq", "wq_b", "w_uk", "wkv", "gamma_ckv")}
    out.update(cos=raw(inp["cos"]), sin=raw(inp["sin"]), cache_index=raw(inp["cache_index"]),
               kv_nope=raw(inp["kv_nope"]) if int8 else bf(inp["kv_nope"]), kv_rope=bf(inp["kv_rope"]),
               kv_scales=raw(inp["kv_scales"]) if int8 else None)
    return out
