"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for sparse MLA attention, for
the Lightning Indexer's top-k selection, for the paged cache writer, for
sliding-window attention, for compressed / sparse compressed attention
(``oracle.compressed``, numpy) and for the MLA Prolog (``oracle.prolog``,
numpy).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA product path never imports it and the
two share no code.  The arithmetic lives in ``mla_oracle.c``,
``indexer_oracle.c``, ``cache_oracle.c`` and ``swa_oracle.c`` (see their
headers for the passages they follow); this
module only compiles them and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "mla_oracle.c"), os.path.join(_HERE, "indexer_oracle.c"),
         os.path.join(_HERE, "cache_oracle.c"), os.path.join(_HERE, "swa_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(map(os.path.getmtime, _SRCS)):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", _LIB_PATH] + _SRCS + ["-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.mla_oracle_fwd.argtypes = [I] * 11 + [P] * 8 + [ctypes.c_double, P, I, P, P, I,
                                                               ctypes.POINTER(ctypes.c_int64)]
        lib.mla_oracle_fwd.restype = I
        lib.mla_oracle_dequant_rows.argtypes = [P, P, ctypes.c_int64, I, P]
        lib.mla_oracle_dequant_rows.restype = None
        lib.mla_oracle_max_threads.argtypes = []
        lib.mla_oracle_max_threads.restype = I
        lib.idx_oracle_scores.argtypes = [I] * 7 + [P] * 5 + [I, P, I, ctypes.POINTER(ctypes.c_int64)]
        lib.idx_oracle_scores.restype = I
        lib.idx_oracle_select.argtypes = [I, I, P, I, P, I, P]
        lib.idx_oracle_select.restype = I
        lib.cache_oracle_write.argtypes = [I, I, ctypes.c_int64, P, P, P, P, P, P, ctypes.POINTER(ctypes.c_int64)]
        lib.cache_oracle_write.restype = I
        lib.swa_oracle_window_lists.argtypes = [I, I, P, I, P]
        lib.swa_oracle_window_lists.restype = I
        _lib = lib
    return _lib


def max_threads() -> int:
    return _load().mla_oracle_max_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(inp: dict, tokens=None, threads: int = 0):
    """Run the oracle on a workload dict (numpy arrays, see workloads.py).

    Returns (out, lse, bad_blocks): out fp64 (n_tokens, n_q, d_nope),
    lse fp64 (n_tokens, n_q).
    """
    lib = _load()
    d = inp["dims"]
    q_nope = np.ascontiguousarray(inp["q_nope"], dtype=np.uint16)
    q_rope = np.ascontiguousarray(inp["q_rope"], dtype=np.uint16)
    kv_int8 = int(d["kv_int8"])
    kv_nope = np.ascontiguousarray(inp["kv_nope"], dtype=np.int8 if kv_int8 else np.uint16)
    kv_rope = np.ascontiguousarray(inp["kv_rope"], dtype=np.uint16)
    kv_scales = None
    if kv_int8:
        kv_scales = np.ascontiguousarray(inp["kv_scales"], dtype=np.float32)
    topk_idx = np.ascontiguousarray(inp["topk_idx"], dtype=np.int32)
    block_table = np.ascontiguousarray(inp["block_table"], dtype=np.int32)
    act_seqs = np.ascontiguousarray(inp["act_seqs"], dtype=np.int32)
    T = d["B"] * d["S1"]
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = int(tok.shape[0])
    out = np.empty((n, d["n_q"], d["d_nope"]), dtype=np.float64)
    lse = np.empty((n, d["n_q"]), dtype=np.float64)
    bad = ctypes.c_int64(0)
    rc = lib.mla_oracle_fwd(d["B"], d["S1"], d["n_q"], d["n_kv"], d["d_nope"], d["d_rope"],
                            d["block_size"], d["num_blocks"], d["max_blocks_per_seq"], d["topk"],
                            kv_int8, _ptr(q_nope), _ptr(q_rope), _ptr(kv_nope), _ptr(kv_rope),
                            _ptr(kv_scales), _ptr(topk_idx), _ptr(block_table), _ptr(act_seqs),
                            float(inp["softmax_scale"]), _ptr(tok), n, _ptr(out), _ptr(lse),
                            int(threads), ctypes.byref(bad))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out, lse, int(bad.value)


def dequant_rows(q8: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The oracle's INT8 -> BF16 dequantisation of whole rows (bf16 bits)."""
    lib = _load()
    q8 = np.ascontiguousarray(q8, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    rows, d_nope = q8.shape
    out = np.empty((rows, d_nope), dtype=np.uint16)
    lib.mla_oracle_dequant_rows(_ptr(q8), _ptr(scales), rows, d_nope, _ptr(out))
    return out


# ------------------------------------------------------------------ Lightning Indexer
def indexer_scores(inp: dict, threads: int = 0):
    """Exact index scores I[t, j] (fp64, (T, ld) with ld = max_blocks_per_seq *
    block_size); -inf where j is not a candidate.  Returns (scores, bad_blocks)."""
    lib = _load()
    d = inp["dims"]
    T = d["B"] * d["S1"]
    ld = d["max_blocks_per_seq"] * d["block_size"]
    scores = np.empty((T, ld), dtype=np.float64)
    bad = ctypes.c_int64(0)
    rc = lib.idx_oracle_scores(d["B"], d["S1"], d["n_heads"], d["head_dim"], d["block_size"], d["num_blocks"],
                               d["max_blocks_per_seq"],
                               _ptr(np.ascontiguousarray(inp["q"], dtype=np.uint16)),
                               _ptr(np.ascontiguousarray(inp["w"], dtype=np.float32)),
                               _ptr(np.ascontiguousarray(inp["k_cache"], dtype=np.uint16)),
                               _ptr(np.ascontiguousarray(inp["block_table"], dtype=np.int32)),
                               _ptr(np.ascontiguousarray(inp["act_seqs"], dtype=np.int32)),
                               ld, _ptr(scores), threads, ctypes.byref(bad))
    if rc != 0:
        raise ValueError(f"idx_oracle_scores rejected the arguments ({rc})")
    return scores, int(bad.value)


def indexer_select(scores, act_seqs, S1: int, topk: int):
    """The selection rule on any scores array (converted exactly to fp64):
    (T, topk) int32, ascending positions, -1 padded."""
    lib = _load()
    sc = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    act = np.ascontiguousarray(act_seqs, dtype=np.int32)
    T, ld = sc.shape
    out = np.empty((T, topk), dtype=np.int32)
    rc = lib.idx_oracle_select(T // S1, S1, _ptr(act), ld, _ptr(sc), topk, _ptr(out))
    if rc != 0:
        raise ValueError(f"idx_oracle_select rejected the arguments ({rc})")
    return out


def cache_write(k_nope, k_rope, cache_index, kv_nope, kv_rope, kv_scales=None, inplace=False):
    """Write rows into copies of the given cache arrays (numpy), or into the
    arrays themselves with ``inplace`` (they must then be C-contiguous of the
    right dtypes): k_nope (T, 512) and k_rope (T, 64) as bf16 bits (uint16),
    cache_index (T,) int64 flat rows; kv_nope (rows, 512) uint16 (bf16) or int8
    (then kv_scales (rows, 4) fp32), kv_rope (rows, 64) uint16.  Returns
    (kv_nope, kv_rope, kv_scales, skipped_bad)."""
    lib = _load()
    kv_int8 = kv_nope.dtype == np.int8
    if inplace:
        kn, kr, ks = kv_nope, kv_rope, (kv_scales if kv_int8 else None)
        assert kn.flags.c_contiguous and kr.flags.c_contiguous and kr.dtype == np.uint16
        assert ks is None or (ks.flags.c_contiguous and ks.dtype == np.float32)
    else:
        kn = np.array(kv_nope, copy=True, order="C")
        kr = np.array(kv_rope, dtype=np.uint16, copy=True, order="C")
        ks = np.array(kv_scales, dtype=np.float32, copy=True, order="C") if kv_int8 else None
    idx = np.ascontiguousarray(cache_index, dtype=np.int64)
    bad = ctypes.c_int64(0)
    rc = lib.cache_oracle_write(int(idx.shape[0]), int(kv_int8), int(kn.shape[0]),
                                _ptr(np.ascontiguousarray(k_nope, dtype=np.uint16)),
                                _ptr(np.ascontiguousarray(k_rope, dtype=np.uint16)), _ptr(idx), _ptr(kn), _ptr(kr),
                                _ptr(ks), ctypes.byref(bad))
    if rc != 0:
        raise ValueError(f"cache_oracle_write rejected the arguments ({rc})")
    return kn, kr, ks, int(bad.value)


def swa_window_lists(act_seqs, S1: int, window: int):
    """Each token's window positions (B*S1, window) int32, -1 where negative."""
    lib = _load()
    act = np.ascontiguousarray(act_seqs, dtype=np.int32)
    B = int(act.shape[0])
    lists = np.empty((B * S1, window), dtype=np.int32)
    if lib.swa_oracle_window_lists(B, S1, _ptr(act), int(window), _ptr(lists)) != 0:
        raise ValueError("swa_oracle_window_lists rejected the arguments")
    return lists


def swa_forward(inp: dict, window: int, tokens=None, threads: int = 0):
    """Sliding-window attention: the window lists, then the attention
    definition over them (``forward`` with top-k = the window)."""
    d = dict(inp["dims"])
    d["topk"] = int(window)
    lists = swa_window_lists(inp["act_seqs"], d["S1"], window)
    return forward(dict(inp, dims=d, topk_idx=lists), tokens=tokens, threads=threads)
