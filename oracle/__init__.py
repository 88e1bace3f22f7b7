"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for sparse MLA attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA product path never imports it and the
two share no code.  The arithmetic lives in ``mla_oracle.c`` (see its header
for the passages it follows); this module only compiles it and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", _LIB_PATH, _SRC, "-lm"]
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
