"""ctypes binding of the C ABI in include/mla_sparse.h, mla_indexer.h,
mla_cache.h and mla_prolog.h.

Argument marshalling only: shapes and dtypes are read off torch tensors, the
device pointers and the current CUDA stream are passed through, and a
negative status becomes an exception.  With the environment variable
MLA_SPARSE_DEBUG set (to anything but "" or "0") every call also synchronises
its stream and raises MlaError when the device status word of its operation
has a bit set (a bad block id, a wait that ran out), instead of leaving it for
a later *_device_status call.  Every step of the computation runs in
the CUDA library; there is no other implementation to fall back to, and a
missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_sparse.so")

MLA_OK = 0
MLA_MODE_DECODE = 0
MLA_MODE_PREFILL = 1
MLA_KV_BF16 = 0
MLA_KV_INT8 = 1
MLA_DEVICE_BAD_BLOCK = 0x1
MLA_DEVICE_TIMEOUT = 0x2

EXPORTED_SYMBOLS = ("mla_sparse_attn_fwd", "mla_swa_fwd", "mla_compressed_attn_fwd", "mla_sparse_last_error", "mla_sparse_device_status",
                    "mla_sparse_get_device_status", "mla_sparse_set_wait_limit_ns", "mla_sparse_launch_count",
                    "mla_sparse_allow_cut_tokens",
                    "mla_sparse_abi_version", "mla_indexer_workspace_bytes", "mla_indexer_topk",
                    "mla_indexer_scores", "mla_indexer_select", "mla_indexer_device_status",
                    "mla_indexer_last_error", "mla_indexer_topk_noalloc", "mla_cache_write",
                    "mla_cache_last_error", "mla_cache_device_status", "mla_prolog_workspace_bytes", "mla_prolog",
                    "mla_prolog_last_error", "mla_prolog_device_status")


class MlaDims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "B", "S1", "n_q", "n_kv", "d_nope", "d_rope", "block_size", "num_blocks", "max_blocks_per_seq",
        "topk", "kv_dtype")]


class MlaCmpCache(ctypes.Structure):
    """mla_cmp_cache: the compressed cache of mla_compressed_attn_fwd."""
    _fields_ = [("nope", ctypes.c_void_p), ("rope", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("ratio", ctypes.c_int32),
                ("sparse_idx", ctypes.c_void_p), ("topk", ctypes.c_int32)]


class IndexerDims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "B", "S1", "n_heads", "head_dim", "block_size", "num_blocks", "max_blocks_per_seq", "topk")]


class PrologDims(ctypes.Structure):
    """mla_prolog_dims."""
    _fields_ = [("T", ctypes.c_int32), ("hidden", ctypes.c_int32), ("q_lora", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("num_rows", ctypes.c_int64), ("kv_int8", ctypes.c_int32),
                ("eps", ctypes.c_float)]


class PrologWeights(ctypes.Structure):
    """mla_prolog_weights (device pointers)."""
    _fields_ = [(name, ctypes.c_void_p) for name in ("wq_a", "gamma_cq", "wq_b", "w_uk", "wkv", "gamma_ckv")]


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"mla_sparse status {status}: {message}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -m mla_sparse_top_gb300.build)")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.mla_sparse_attn_fwd.argtypes = [ctypes.POINTER(MlaDims)] + [vp] * 10 + [ctypes.c_float, ctypes.c_int32, vp]
    lib.mla_sparse_attn_fwd.restype = ctypes.c_int
    lib.mla_swa_fwd.argtypes = [ctypes.POINTER(MlaDims)] + [vp] * 7 + [ctypes.c_int32, vp, vp, ctypes.c_float,
                                                                        ctypes.c_int32, vp]
    lib.mla_swa_fwd.restype = ctypes.c_int
    lib.mla_compressed_attn_fwd.argtypes = [ctypes.POINTER(MlaDims)] + [vp] * 6 + [ctypes.POINTER(MlaCmpCache), vp,
                                                                                   ctypes.c_int32, vp, vp,
                                                                                   ctypes.c_float, ctypes.c_int32, vp]
    lib.mla_compressed_attn_fwd.restype = ctypes.c_int
    lib.mla_sparse_last_error.argtypes = []
    lib.mla_sparse_last_error.restype = ctypes.c_char_p
    lib.mla_sparse_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]
    lib.mla_sparse_device_status.restype = ctypes.c_int
    lib.mla_sparse_get_device_status.argtypes = [vp]
    lib.mla_sparse_get_device_status.restype = ctypes.c_int
    lib.mla_sparse_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.mla_sparse_set_wait_limit_ns.restype = ctypes.c_int
    lib.mla_sparse_launch_count.argtypes = []
    lib.mla_sparse_launch_count.restype = ctypes.c_uint64
    lib.mla_sparse_allow_cut_tokens.argtypes = [ctypes.c_int32]
    lib.mla_sparse_allow_cut_tokens.restype = None
    lib.mla_sparse_abi_version.argtypes = []
    lib.mla_sparse_abi_version.restype = ctypes.c_int32
    lib.mla_indexer_workspace_bytes.argtypes = [ctypes.POINTER(IndexerDims)]
    lib.mla_indexer_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_indexer_topk.argtypes = [ctypes.POINTER(IndexerDims)] + [vp] * 7 + [ctypes.c_size_t, vp]
    lib.mla_indexer_topk.restype = ctypes.c_int
    lib.mla_indexer_scores.argtypes = [ctypes.POINTER(IndexerDims)] + [vp] * 6 + [ctypes.c_size_t, vp]
    lib.mla_indexer_scores.restype = ctypes.c_int
    lib.mla_indexer_select.argtypes = [ctypes.POINTER(IndexerDims)] + [vp] * 4
    lib.mla_indexer_select.restype = ctypes.c_int
    lib.mla_indexer_topk_noalloc.argtypes = [ctypes.POINTER(IndexerDims)] + [vp] * 7
    lib.mla_indexer_topk_noalloc.restype = ctypes.c_int
    lib.mla_cache_write.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32] + [vp] * 7
    lib.mla_cache_write.restype = ctypes.c_int
    lib.mla_cache_last_error.argtypes = []
    lib.mla_cache_last_error.restype = ctypes.c_char_p
    lib.mla_cache_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]
    lib.mla_cache_device_status.restype = ctypes.c_int
    lib.mla_indexer_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]
    lib.mla_indexer_device_status.restype = ctypes.c_int
    lib.mla_indexer_last_error.argtypes = []
    lib.mla_indexer_last_error.restype = ctypes.c_char_p
    lib.mla_prolog_workspace_bytes.argtypes = [ctypes.POINTER(PrologDims)]
    lib.mla_prolog_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_prolog.argtypes = [ctypes.POINTER(PrologDims), vp, ctypes.POINTER(PrologWeights)] + [vp] * 9 + [
        ctypes.c_size_t, vp]
    lib.mla_prolog.restype = ctypes.c_int
    lib.mla_prolog_last_error.argtypes = []
    lib.mla_prolog_last_error.restype = ctypes.c_char_p
    lib.mla_prolog_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]
    lib.mla_prolog_device_status.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != MLA_OK:
        raise MlaError(status, load_library().mla_sparse_last_error().decode())


def debug_enabled() -> bool:
    """True when MLA_SPARSE_DEBUG asks for a status check after every call."""
    return os.environ.get("MLA_SPARSE_DEBUG", "") not in ("", "0")


def _debug_status(read_status, what: str, stream):
    """Under MLA_SPARSE_DEBUG: synchronise, read and clear the operation's
    status word, raise MlaError(MLA_ERR_DEVICE_STATUS) if a bit was set."""
    if not debug_enabled():
        return
    flags = read_status(clear=True, stream=stream)
    if flags:
        raise MlaError(-7, f"{what}: device status {flags:#x} after the call (MLA_SPARSE_DEBUG)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dims_from_workload(d: dict) -> MlaDims:
    """MlaDims from a dimension dict with the header's field names (kv_int8 flag)."""
    return MlaDims(B=d["B"], S1=d["S1"], n_q=d["n_q"], n_kv=d["n_kv"], d_nope=d["d_nope"], d_rope=d["d_rope"],
                   block_size=d["block_size"], num_blocks=d["num_blocks"], max_blocks_per_seq=d["max_blocks_per_seq"],
                   topk=d["topk"], kv_dtype=MLA_KV_INT8 if d["kv_int8"] else MLA_KV_BF16)


def make_dims(q_nope, kv_nope, topk_idx, block_table, kv_int8: bool, S1: int) -> MlaDims:
    T, n_q, d_nope = q_nope.shape
    if T % S1:
        raise ValueError("q_nope's leading dim must be B*S1")
    rows = kv_nope.shape[0]
    return MlaDims(B=T // S1, S1=S1, n_q=n_q, n_kv=1, d_nope=d_nope, d_rope=64, block_size=128,
                   num_blocks=rows // 128, max_blocks_per_seq=block_table.shape[1], topk=topk_idx.shape[1],
                   kv_dtype=MLA_KV_INT8 if kv_int8 else MLA_KV_BF16)


def mla_sparse_attn_fwd(q_nope, q_rope, kv_nope, kv_rope, kv_scales, topk_idx, block_table, act_seqs, out,
                        lse=None, softmax_scale=None, mode: int | str = MLA_MODE_DECODE, S1: int = 1,
                        stream=None, dims: MlaDims | None = None):
    """Enqueue one call of the C entry point with the same name.

    q_nope (B*S1, n_q, 512) bf16, q_rope (B*S1, n_q, 64) bf16, kv_nope
    (rows, 512) bf16|int8, kv_rope (rows, 64) bf16, kv_scales (rows, 4) fp32 or
    None, topk_idx (B*S1, topk) int32, block_table (B, W) int32, act_seqs (B,)
    int32, out (B*S1, n_q, 512) bf16, lse (B*S1, n_q) fp32 or None.
    """
    lib = load_library()
    kv_int8 = kv_nope.dtype == torch.int8
    if dims is None:
        dims = make_dims(q_nope, kv_nope, topk_idx, block_table, kv_int8, S1)
    if isinstance(mode, str):
        mode = {"decode": MLA_MODE_DECODE, "prefill": MLA_MODE_PREFILL}[mode]
    if softmax_scale is None:
        softmax_scale = (dims.d_nope + dims.d_rope) ** -0.5
    st = lib.mla_sparse_attn_fwd(ctypes.byref(dims), _ptr(q_nope), _ptr(q_rope), _ptr(kv_nope), _ptr(kv_rope),
                                 _ptr(kv_scales if kv_int8 else None), _ptr(topk_idx), _ptr(block_table),
                                 _ptr(act_seqs), _ptr(out), _ptr(lse), ctypes.c_float(softmax_scale),
                                 ctypes.c_int32(int(mode)), _stream_handle(stream))
    _check(st)
    _debug_status(device_status, "mla_sparse_attn_fwd", stream)
    return out, lse


def mla_swa_fwd(q_nope, q_rope, kv_nope, kv_rope, kv_scales, block_table, act_seqs, out, lse=None, *,
                window: int, softmax_scale=None, mode: int | str = MLA_MODE_DECODE, S1: int = 1, stream=None,
                dims: MlaDims | None = None):
    """Enqueue one call of the C entry point with the same name: sliding-window
    attention, token (b, s) at position act_seqs[b] - S1 + s attending to the
    `window` positions ending at its own.  Tensors as mla_sparse_attn_fwd
    without topk_idx."""
    lib = load_library()
    kv_int8 = kv_nope.dtype == torch.int8
    if dims is None:
        T, n_q, d_nope = q_nope.shape
        dims = MlaDims(B=T // S1, S1=S1, n_q=n_q, n_kv=1, d_nope=d_nope, d_rope=64, block_size=128,
                       num_blocks=kv_nope.shape[0] // 128, max_blocks_per_seq=block_table.shape[1], topk=window,
                       kv_dtype=MLA_KV_INT8 if kv_int8 else MLA_KV_BF16)
    if isinstance(mode, str):
        mode = {"decode": MLA_MODE_DECODE, "prefill": MLA_MODE_PREFILL}[mode]
    if softmax_scale is None:
        softmax_scale = (dims.d_nope + dims.d_rope) ** -0.5
    st = lib.mla_swa_fwd(ctypes.byref(dims), _ptr(q_nope), _ptr(q_rope), _ptr(kv_nope), _ptr(kv_rope),
                         _ptr(kv_scales if kv_int8 else None), _ptr(block_table), _ptr(act_seqs),
                         ctypes.c_int32(int(window)), _ptr(out), _ptr(lse), ctypes.c_float(softmax_scale),
                         ctypes.c_int32(int(mode)), _stream_handle(stream))
    _check(st)
    _debug_status(device_status, "mla_swa_fwd", stream)
    return out, lse


def mla_compressed_attn_fwd(q_nope, q_rope, kv_nope, kv_rope, kv_scales, block_table, cmp_nope, cmp_rope,
                            cmp_scales, cmp_block_table, act_seqs, out, lse=None, *, window: int, cmp_ratio: int,
                            cmp_idx=None, softmax_scale=None, mode: int | str = MLA_MODE_DECODE, S1: int = 1,
                            stream=None, dims: MlaDims | None = None):
    """Enqueue one call of the C entry point with the same name: each token's
    window of the original cache plus the compressed cache's visible entries
    (CFA, cmp_idx None) or the visible entries of cmp_idx (SCFA, (B*S1, K)
    int32).  The compressed cache has the original layout and dtype."""
    lib = load_library()
    kv_int8 = kv_nope.dtype == torch.int8
    if dims is None:
        T, n_q, d_nope = q_nope.shape
        dims = MlaDims(B=T // S1, S1=S1, n_q=n_q, n_kv=1, d_nope=d_nope, d_rope=64, block_size=128,
                       num_blocks=kv_nope.shape[0] // 128, max_blocks_per_seq=block_table.shape[1], topk=window,
                       kv_dtype=MLA_KV_INT8 if kv_int8 else MLA_KV_BF16)
    if isinstance(mode, str):
        mode = {"decode": MLA_MODE_DECODE, "prefill": MLA_MODE_PREFILL}[mode]
    if softmax_scale is None:
        softmax_scale = (dims.d_nope + dims.d_rope) ** -0.5
    cmp = MlaCmpCache(nope=_ptr(cmp_nope), rope=_ptr(cmp_rope), scales=_ptr(cmp_scales if kv_int8 else None),
                      block_table=_ptr(cmp_block_table), num_blocks=cmp_nope.shape[0] // 128,
                      max_blocks_per_seq=cmp_block_table.shape[1], ratio=int(cmp_ratio), sparse_idx=_ptr(cmp_idx),
                      topk=int(cmp_idx.shape[1]) if cmp_idx is not None else 0)
    st = lib.mla_compressed_attn_fwd(ctypes.byref(dims), _ptr(q_nope), _ptr(q_rope), _ptr(kv_nope), _ptr(kv_rope),
                                     _ptr(kv_scales if kv_int8 else None), _ptr(block_table), ctypes.byref(cmp),
                                     _ptr(act_seqs), ctypes.c_int32(int(window)), _ptr(out), _ptr(lse),
                                     ctypes.c_float(softmax_scale), ctypes.c_int32(int(mode)),
                                     _stream_handle(stream))
    _check(st)
    _debug_status(device_status, "mla_compressed_attn_fwd", stream)
    return out, lse


def device_status(clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return (and by default clear) the status bits."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    st = lib.mla_sparse_device_status(_stream_handle(stream), ctypes.byref(flags), 1 if clear else 0)
    if st not in (MLA_OK, -7):
        _check(st)
    return int(flags.value)


def abi_version() -> int:
    return int(load_library().mla_sparse_abi_version())


def set_wait_limit_ns(ns: int) -> None:
    """Bound of every device-side wait of later attention launches."""
    _check(load_library().mla_sparse_set_wait_limit_ns(int(ns)))


DEFAULT_WAIT_LIMIT_NS = 500 * 1000 * 1000


def launch_count() -> int:
    """Kernel launches the attention entry points have enqueued in this process."""
    return int(load_library().mla_sparse_launch_count())


def allow_cut_tokens(allow: bool) -> None:
    """Whether later attention calls may cut tokens between clusters (the default)."""
    load_library().mla_sparse_allow_cut_tokens(1 if allow else 0)


# ------------------------------------------------------------------ Lightning Indexer
def _check_idx(status: int):
    if status != MLA_OK:
        raise MlaError(status, load_library().mla_indexer_last_error().decode())


def indexer_dims_from_workload(d: dict) -> IndexerDims:
    return IndexerDims(**{f: int(d[f]) for f, _ in IndexerDims._fields_})


def mla_indexer_workspace_bytes(dims: IndexerDims) -> int:
    return int(load_library().mla_indexer_workspace_bytes(ctypes.byref(dims)))


def mla_indexer_topk(q, w, k_cache, block_table, act_seqs, topk_idx, workspace, *, dims: IndexerDims, stream=None):
    """Enqueue one call of the C entry point with the same name.

    q (B*S1, H, 128) bf16, w (B*S1, H) fp32, k_cache (rows, 128) bf16,
    block_table (B, W) int32, act_seqs (B,) int32, topk_idx (B*S1, topk) int32
    (output), workspace: a device tensor of at least
    mla_indexer_workspace_bytes(dims) bytes (holds the fp32 scores [B*S1, W*128]
    on return).
    """
    lib = load_library()
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.mla_indexer_topk(ctypes.byref(dims), _ptr(q), _ptr(w), _ptr(k_cache), _ptr(block_table), _ptr(act_seqs),
                              _ptr(topk_idx), _ptr(workspace), ctypes.c_size_t(nbytes), _stream_handle(stream))
    _check_idx(st)
    _debug_status(indexer_device_status, "mla_indexer_topk", stream)
    return topk_idx


def mla_indexer_scores(q, w, k_cache, block_table, act_seqs, scores, *, dims: IndexerDims, stream=None):
    """Enqueue the score phase alone (C entry point of the same name); scores is
    a device tensor of at least mla_indexer_workspace_bytes(dims) bytes."""
    lib = load_library()
    nbytes = scores.numel() * scores.element_size()
    st = lib.mla_indexer_scores(ctypes.byref(dims), _ptr(q), _ptr(w), _ptr(k_cache), _ptr(block_table),
                                _ptr(act_seqs), _ptr(scores), ctypes.c_size_t(nbytes), _stream_handle(stream))
    _check_idx(st)
    _debug_status(indexer_device_status, "mla_indexer_scores", stream)
    return scores


def mla_indexer_select(scores, act_seqs, topk_idx, *, dims: IndexerDims, stream=None):
    """Enqueue the selection phase alone (C entry point of the same name) on
    fp32 scores [B*S1, W*128]."""
    lib = load_library()
    st = lib.mla_indexer_select(ctypes.byref(dims), _ptr(scores), _ptr(act_seqs), _ptr(topk_idx),
                                _stream_handle(stream))
    _check_idx(st)
    _debug_status(indexer_device_status, "mla_indexer_select", stream)
    return topk_idx


def mla_indexer_topk_noalloc(q, w, k_cache, block_table, act_seqs, topk_idx, *, dims: IndexerDims, stream=None):
    """Enqueue one call of the C entry point with the same name: the indexer
    and top-k with the scores in the library's fixed scratch (no workspace,
    nothing allocated; at most 2,097,152 scores per call, and calls that
    overlap in time race on the scratch)."""
    lib = load_library()
    st = lib.mla_indexer_topk_noalloc(ctypes.byref(dims), _ptr(q), _ptr(w), _ptr(k_cache), _ptr(block_table),
                                      _ptr(act_seqs), _ptr(topk_idx), _stream_handle(stream))
    _check_idx(st)
    _debug_status(indexer_device_status, "mla_indexer_topk_noalloc", stream)
    return topk_idx


def indexer_device_status(clear: bool = True, stream=None) -> int:
    lib = load_library()
    flags = ctypes.c_uint32(0)
    st = lib.mla_indexer_device_status(_stream_handle(stream), ctypes.byref(flags), 1 if clear else 0)
    if st not in (MLA_OK, -7):
        _check_idx(st)
    return int(flags.value)


# ------------------------------------------------------------------ paged cache writer
def mla_cache_write(k_nope, k_rope, cache_index, kv_nope, kv_rope, kv_scales=None, *, stream=None):
    """Enqueue one call of the C entry point with the same name: k_nope (T, 512)
    and k_rope (T, 64) bf16, cache_index (T,) int64 flat rows; kv_nope (rows,
    512) bf16 or int8 (then kv_scales (rows, 4) fp32) and kv_rope (rows, 64)
    bf16 are updated in place."""
    lib = load_library()
    kv_int8 = 1 if kv_nope.element_size() == 1 else 0
    st = lib.mla_cache_write(int(cache_index.shape[0]), int(kv_nope.shape[0]), kv_int8, _ptr(k_nope), _ptr(k_rope),
                             _ptr(cache_index), _ptr(kv_nope), _ptr(kv_rope), _ptr(kv_scales),
                             _stream_handle(stream))
    if st != MLA_OK:
        raise MlaError(st, lib.mla_cache_last_error().decode())
    _debug_status(cache_device_status, "mla_cache_write", stream)


def cache_device_status(clear: bool = True, stream=None) -> int:
    lib = load_library()
    flags = ctypes.c_uint32(0)
    st = lib.mla_cache_device_status(_stream_handle(stream), ctypes.byref(flags), 1 if clear else 0)
    if st not in (MLA_OK, -7):
        raise MlaError(st, lib.mla_cache_last_error().decode())
    return int(flags.value)


# ------------------------------------------------------------------ MLA Prolog
PROLOG_EPS = 1e-6


def prolog_dims(x, wq_a, wq_b, kv_nope, eps: float = PROLOG_EPS) -> PrologDims:
    """PrologDims read off the tensors: x (T, hidden), wq_a (hidden, q_lora),
    wq_b (q_lora, H * 192), kv_nope (rows, 512)."""
    return PrologDims(T=int(x.shape[0]), hidden=int(x.shape[1]), q_lora=int(wq_a.shape[1]),
                      n_heads=int(wq_b.shape[1]) // 192, num_rows=int(kv_nope.shape[0]),
                      kv_int8=1 if kv_nope.element_size() == 1 else 0, eps=float(eps))


def mla_prolog_workspace_bytes(dims: PrologDims) -> int:
    return int(load_library().mla_prolog_workspace_bytes(ctypes.byref(dims)))


def mla_prolog(x, wq_a, gamma_cq, wq_b, w_uk, wkv, gamma_ckv, cos, sin, cache_index, q_nope, q_rope, kv_nope,
               kv_rope, kv_scales, workspace, *, eps: float = PROLOG_EPS, dims: PrologDims | None = None,
               stream=None):
    """Enqueue one call of the C entry point with the same name.

    x (T, hidden) bf16; weights bf16: wq_a (hidden, q_lora), gamma_cq (q_lora,),
    wq_b (q_lora, H*192), w_uk (H, 128, 512), wkv (hidden, 576), gamma_ckv
    (576,); cos / sin (T, 32) fp32; cache_index (T,) int64; outputs q_nope
    (T, H, 512) and q_rope (T, H, 64) bf16; the cache kv_nope (rows, 512) bf16
    or int8 (then kv_scales (rows, 4) fp32) and kv_rope (rows, 64) bf16 is
    updated in place; workspace: a device tensor of at least
    mla_prolog_workspace_bytes(dims) bytes."""
    lib = load_library()
    if dims is None:
        dims = prolog_dims(x, wq_a, wq_b, kv_nope, eps)
    wts = PrologWeights(wq_a=_ptr(wq_a), gamma_cq=_ptr(gamma_cq), wq_b=_ptr(wq_b), w_uk=_ptr(w_uk), wkv=_ptr(wkv),
                        gamma_ckv=_ptr(gamma_ckv))
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.mla_prolog(ctypes.byref(dims), _ptr(x), ctypes.byref(wts), _ptr(cos), _ptr(sin), _ptr(cache_index),
                        _ptr(q_nope), _ptr(q_rope), _ptr(kv_nope), _ptr(kv_rope),
                        _ptr(kv_scales if dims.kv_int8 else None), _ptr(workspace), ctypes.c_size_t(nbytes),
                        _stream_handle(stream))
    if st != MLA_OK:
        raise MlaError(st, lib.mla_prolog_last_error().decode())
    _debug_status(prolog_device_status, "mla_prolog", stream)
    return q_nope, q_rope


def prolog_device_status(clear: bool = True, stream=None) -> int:
    lib = load_library()
    flags = ctypes.c_uint32(0)
    st = lib.mla_prolog_device_status(_stream_handle(stream), ctypes.byref(flags), 1 if clear else 0)
    if st not in (MLA_OK, -7):
        raise MlaError(st, lib.mla_prolog_last_error().decode())
    return int(flags.value)
