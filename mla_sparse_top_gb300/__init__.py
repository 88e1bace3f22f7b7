"""GB300-native sparse MLA attention over a paged KV cache, the Lightning
Indexer + top-k that selects its entries, the writer that puts new rows into
that cache (bf16 or INT8), and the MLA Prolog that produces the absorbed query
and the new cache rows from hidden states.

The computation lives in ``libmla_sparse.so`` (CUDA for sm_103a, C ABI in
``include/mla_sparse.h``); this package builds it in-tree and exposes it
through a thin ctypes binding with the same entry-point names.
"""
from .binding import (MLA_DEVICE_BAD_BLOCK, MlaCmpCache, cache_device_status, mla_cache_write,
                      mla_compressed_attn_fwd, mla_swa_fwd, MLA_DEVICE_TIMEOUT, MLA_KV_BF16, MLA_KV_INT8, MLA_MODE_DECODE,
                      MLA_MODE_PREFILL, IndexerDims, MlaDims, MlaError, abi_version, device_status, dims_from_workload,
                      indexer_device_status, indexer_dims_from_workload, load_library, mla_indexer_scores,
                      mla_indexer_select, mla_indexer_topk, mla_indexer_topk_noalloc, mla_indexer_workspace_bytes,
                      mla_sparse_attn_fwd, set_wait_limit_ns, DEFAULT_WAIT_LIMIT_NS, launch_count, allow_cut_tokens, PrologDims, PrologWeights, mla_prolog, mla_prolog_workspace_bytes,
                      prolog_device_status, prolog_dims)

__all__ = ["mla_sparse_attn_fwd", "mla_swa_fwd", "mla_compressed_attn_fwd", "MlaCmpCache", "mla_cache_write", "cache_device_status", "device_status", "abi_version", "set_wait_limit_ns", "DEFAULT_WAIT_LIMIT_NS", "launch_count", "allow_cut_tokens", "load_library", "MlaDims", "MlaError", "dims_from_workload",
           "mla_indexer_topk", "mla_indexer_topk_noalloc", "mla_indexer_scores", "mla_indexer_select", "mla_indexer_workspace_bytes", "indexer_device_status", "indexer_dims_from_workload",
           "IndexerDims", "PrologDims", "PrologWeights", "mla_prolog", "mla_prolog_workspace_bytes",
           "prolog_device_status", "prolog_dims",
           "MLA_MODE_DECODE", "MLA_MODE_PREFILL", "MLA_KV_BF16", "MLA_KV_INT8", "MLA_DEVICE_BAD_BLOCK",
           "MLA_DEVICE_TIMEOUT"]
