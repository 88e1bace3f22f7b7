"""Host-side checks of the C ABI: the library builds, loads, exports every
function include/*.h declares, and rejects bad arguments before touching the
GPU (every case below fails validation, so no CUDA call runs)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", "mla_sparse.h"), os.path.join(ROOT, "include", "mla_indexer.h"),
           os.path.join(ROOT, "include", "mla_cache.h"), os.path.join(ROOT, "include", "mla_prolog.h")]


@pytest.fixture(scope="module")
def lib():
    from mla_sparse_top_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(mla_(?:sparse|indexer|cache|swa|compressed|prolog)(?:_\w+)?)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"mla_sparse_attn_fwd", "mla_sparse_last_error", "mla_sparse_device_status",
            "mla_sparse_abi_version", "mla_indexer_topk", "mla_indexer_workspace_bytes",
            "mla_indexer_device_status", "mla_indexer_last_error", "mla_indexer_scores",
            "mla_indexer_select", "mla_indexer_topk_noalloc", "mla_cache_write", "mla_cache_last_error",
            "mla_cache_device_status", "mla_swa_fwd", "mla_compressed_attn_fwd", "mla_prolog",
            "mla_prolog_workspace_bytes", "mla_prolog_last_error", "mla_prolog_device_status",
            "mla_sparse_get_device_status", "mla_sparse_set_wait_limit_ns", "mla_sparse_launch_count", "mla_sparse_allow_cut_tokens"} <= set(names)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    from mla_sparse_top_gb300 import binding
    assert set(binding.EXPORTED_SYMBOLS) == set(declared_functions())
    assert lib.mla_sparse_abi_version() == 202


@pytest.mark.parametrize("ns, expect", [(0, -2), (999, -2), (60 * 10**9 + 1, -2), (1000, 0), (500 * 10**6, 0)])
def test_wait_limit_range(lib, ns, expect):
    lib.mla_sparse_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    assert lib.mla_sparse_set_wait_limit_ns(ns) == expect
    lib.mla_sparse_set_wait_limit_ns(500 * 10**6)


def _dims(**kw):
    from mla_sparse_top_gb300.binding import MlaDims
    d = dict(B=2, S1=2, n_q=128, n_kv=1, d_nope=512, d_rope=64, block_size=128, num_blocks=16,
             max_blocks_per_seq=8, topk=2048, kv_dtype=0)
    d.update(kw)
    return MlaDims(**d)


def _call(lib, dims, ptrs=None, scales=None, scale=0.04, mode=0):
    p = ptrs if ptrs is not None else [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    q_nope, q_rope, kv_nope, kv_rope, topk, bt, act, out, lse = p
    return lib.mla_sparse_attn_fwd(None if dims is None else ctypes.byref(dims), q_nope, q_rope, kv_nope,
                                   kv_rope, scales, topk, bt, act, out, lse, ctypes.c_float(scale),
                                   ctypes.c_int32(mode), None)


@pytest.mark.parametrize("case,expect", [
    ("null_dims", -1), ("null_q", -1), ("bad_dtype", -3), ("int8_no_scales", -3), ("n_q_zero", -2),
    ("n_q_big", -2), ("n_kv_2", -4), ("d_nope_256", -4), ("block_64", -4), ("topk_zero", -2),
    ("mode_bad", -2), ("scale_nan", -2), ("misaligned_kv", -5), ("misaligned_topk", -5), ("batch_zero", -2),
    ("blocks_huge", -2),
])
def test_argument_errors_are_reported_before_launch(lib, case, expect):
    dims = _dims()
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    scales = None
    scale = 0.04
    mode = 0
    if case == "null_dims":
        dims = None
    elif case == "null_q":
        ptrs[0] = None
    elif case == "bad_dtype":
        dims = _dims(kv_dtype=7)
    elif case == "int8_no_scales":
        dims = _dims(kv_dtype=1)
    elif case == "n_q_zero":
        dims = _dims(n_q=0)
    elif case == "n_q_big":
        dims = _dims(n_q=129)
    elif case == "n_kv_2":
        dims = _dims(n_kv=2)
    elif case == "d_nope_256":
        dims = _dims(d_nope=256)
    elif case == "block_64":
        dims = _dims(block_size=64)
    elif case == "topk_zero":
        dims = _dims(topk=0)
    elif case == "mode_bad":
        mode = 5
    elif case == "scale_nan":
        scale = float("nan")
    elif case == "misaligned_kv":
        ptrs[2] = ctypes.c_void_p(0x20008)
    elif case == "misaligned_topk":
        ptrs[4] = ctypes.c_void_p(0x50002)
    elif case == "batch_zero":
        dims = _dims(B=0)
    elif case == "blocks_huge":
        dims = _dims(num_blocks=1 << 24)
    st = _call(lib, dims, ptrs, scales, scale, mode)
    assert st == expect
    assert lib.mla_sparse_last_error().decode() != ""


def test_binding_fails_loudly_without_library(tmp_path):
    from mla_sparse_top_gb300 import binding
    with pytest.raises(RuntimeError):
        binding.ctypes  # noqa: B018  (module is importable)
        saved = binding._lib
        binding._lib = None
        try:
            binding.load_library(str(tmp_path / "missing.so"))
        finally:
            binding._lib = saved


# ------------------------------------------------------------------ Lightning Indexer
def _idims(**kw):
    from mla_sparse_top_gb300.binding import IndexerDims
    d = dict(B=2, S1=2, n_heads=64, head_dim=128, block_size=128, num_blocks=16, max_blocks_per_seq=8, topk=64)
    d.update(kw)
    return IndexerDims(**d)


def test_indexer_workspace_size(lib):
    d = _idims()
    assert lib.mla_indexer_workspace_bytes(ctypes.byref(d)) == 2 * 2 * 8 * 128 * 4
    assert lib.mla_indexer_workspace_bytes(ctypes.byref(_idims(n_heads=24))) == 0
    assert lib.mla_indexer_workspace_bytes(None) == 0


@pytest.mark.parametrize("case,expect", [
    ("null_dims", -1), ("null_q", -1), ("null_ws", -1), ("heads_24", -4), ("heads_x_s1_big", -4), ("dim_64", -4),
    ("block_64", -4), ("topk_zero", -2), ("batch_zero", -2), ("ws_small", -2), ("misaligned_q", -5),
    ("misaligned_ws", -5),
])
def test_indexer_argument_errors_are_reported_before_launch(lib, case, expect):
    d = _idims()
    ptr = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(7)]
    q, w, k, bt, act, topk, ws = ptr
    ws_bytes = 2 * 2 * 8 * 128 * 4
    dims = ctypes.byref(d)
    if case == "null_dims":
        dims = None
    elif case == "null_q":
        q = None
    elif case == "null_ws":
        ws = None
    elif case == "heads_24":
        d.n_heads = 24
    elif case == "heads_x_s1_big":
        d.n_heads, d.S1 = 256, 2
    elif case == "dim_64":
        d.head_dim = 64
    elif case == "block_64":
        d.block_size = 64
    elif case == "topk_zero":
        d.topk = 0
    elif case == "batch_zero":
        d.B = 0
    elif case == "ws_small":
        ws_bytes -= 4
    elif case == "misaligned_q":
        q = ctypes.c_void_p(0x100008)
    elif case == "misaligned_ws":
        ws = ctypes.c_void_p(0x100080)
    st = lib.mla_indexer_topk(dims, q, w, k, bt, act, topk, ws, ctypes.c_size_t(ws_bytes), None)
    assert st == expect, (case, st, lib.mla_indexer_last_error())
    assert lib.mla_indexer_last_error()


@pytest.mark.parametrize("case,expect", [("null_scores", -1), ("small", -2), ("misaligned", -5), ("heads_24", -4)])
def test_indexer_score_phase_argument_errors(lib, case, expect):
    d = _idims()
    q, w, k, bt, act, sc = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(6)]
    nbytes = 2 * 2 * 8 * 128 * 4
    if case == "null_scores":
        sc = None
    elif case == "small":
        nbytes = 16
    elif case == "misaligned":
        sc = ctypes.c_void_p(0x100040)
    elif case == "heads_24":
        d.n_heads = 24
    st = lib.mla_indexer_scores(ctypes.byref(d), q, w, k, bt, act, sc, ctypes.c_size_t(nbytes), None)
    assert st == expect, (case, st, lib.mla_indexer_last_error())


@pytest.mark.parametrize("case,expect", [("null_out", -1), ("misaligned", -5), ("topk_zero", -2)])
def test_indexer_select_phase_argument_errors(lib, case, expect):
    d = _idims()
    sc, act, out = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(3)]
    if case == "null_out":
        out = None
    elif case == "misaligned":
        sc = ctypes.c_void_p(0x100002)
    elif case == "topk_zero":
        d.topk = 0
    st = lib.mla_indexer_select(ctypes.byref(d), sc, act, out, None)
    assert st == expect, (case, st, lib.mla_indexer_last_error())


def test_indexer_noalloc_rejects_oversize_before_any_cuda_call(lib):
    d = _idims(B=64, S1=2, max_blocks_per_seq=129)  # 64 * 2 * 129 * 128 scores > 2 Mi
    p = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(7)]
    st = lib.mla_indexer_topk_noalloc(ctypes.byref(d), *p, None)
    assert st == -2
    msg = lib.mla_indexer_last_error().decode()
    assert "exceed" in msg and "mla_indexer_topk" in msg


@pytest.mark.parametrize("case,expect", [("negative_T", -2), ("no_rows", -2), ("bad_mode", -2), ("null_src", -1),
                                         ("int8_no_scales", -1), ("misaligned_cache", -5), ("misaligned_index", -5),
                                         ("empty", 0)])
def test_cache_write_argument_errors_are_reported_before_launch(lib, case, expect):
    T, rows, mode = 4, 256, 1
    p = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(6)]  # k_nope k_rope index kv_nope kv_rope kv_scales
    if case == "negative_T":
        T = -1
    elif case == "no_rows":
        rows = 0
    elif case == "bad_mode":
        mode = 2
    elif case == "null_src":
        p[0] = None
    elif case == "int8_no_scales":
        p[5] = None
    elif case == "misaligned_cache":
        p[3] = ctypes.c_void_p(0x100004)
    elif case == "misaligned_index":
        p[2] = ctypes.c_void_p(0x100004)
    elif case == "empty":
        T = 0
    st = lib.mla_cache_write(T, ctypes.c_int64(rows), mode, *p, None)
    assert st == expect, (case, st, lib.mla_cache_last_error())
    if expect != 0:
        assert lib.mla_cache_last_error()


@pytest.mark.parametrize("window,expect", [(0, -2), (-3, -2)])
def test_swa_rejects_a_window_below_one(lib, window, expect):
    from mla_sparse_top_gb300.binding import MlaDims
    d = MlaDims(B=2, S1=2, n_q=128, n_kv=1, d_nope=512, d_rope=64, block_size=128, num_blocks=8,
                max_blocks_per_seq=4, topk=0, kv_dtype=0)
    p = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(7)]
    st = lib.mla_swa_fwd(ctypes.byref(d), *p, window, ctypes.c_void_p(0x900000), None, ctypes.c_float(0.04), 0, None)
    assert st == expect and b"window" in lib.mla_sparse_last_error()


@pytest.mark.parametrize("case,expect", [("no_cmp", -1), ("window0", -2), ("ratio0", -2), ("scfa_topk0", -2),
                                         ("int8_no_scales", -1), ("big_cache", -2), ("misaligned", -5)])
def test_compressed_attn_argument_errors(lib, case, expect):
    from mla_sparse_top_gb300.binding import MlaCmpCache, MlaDims
    d = MlaDims(B=2, S1=2, n_q=128, n_kv=1, d_nope=512, d_rope=64, block_size=128, num_blocks=8,
                max_blocks_per_seq=4, topk=0, kv_dtype=0)
    P = lambda k: ctypes.c_void_p(0x100000 * k)
    cmp = MlaCmpCache(nope=0x900000, rope=0xA00000, scales=None, block_table=0xB00000, num_blocks=2,
                      max_blocks_per_seq=1, ratio=4, sparse_idx=None, topk=0)
    window = 16
    cref = ctypes.byref(cmp)
    if case == "no_cmp":
        cref = None
    elif case == "window0":
        window = 0
    elif case == "ratio0":
        cmp.ratio = 0
    elif case == "scfa_topk0":
        cmp.sparse_idx = 0xC00000
    elif case == "int8_no_scales":
        d.kv_dtype = 1
    elif case == "big_cache":
        cmp.num_blocks = 1 << 23
    elif case == "misaligned":
        cmp.nope = 0x900004
    st = lib.mla_compressed_attn_fwd(ctypes.byref(d), P(1), P(2), P(3), P(4), P(5) if case == "int8_no_scales" else None,
                                     P(6), cref, P(7), window, P(8), None, ctypes.c_float(0.04), 0, None)
    assert st == expect, (case, st, lib.mla_sparse_last_error())


@pytest.mark.parametrize("case,expect", [
    ("null_dims", -1), ("hidden_7", -2), ("q_lora_0", -2), ("heads_0", -2), ("eps_0", -2), ("rows_0", -2),
    ("int8_2", -2), ("null_x", -1), ("null_weight", -1), ("int8_no_scales", -1), ("misaligned_x", -5),
    ("misaligned_gamma", -5), ("misaligned_ws", -5), ("small_ws", -2), ("empty", 0)])
def test_prolog_argument_errors_are_reported_before_launch(lib, case, expect):
    from mla_sparse_top_gb300.binding import PrologDims, PrologWeights
    d = PrologDims(T=4, hidden=64, q_lora=32, n_heads=2, num_rows=256, kv_int8=1, eps=1e-6)
    P = lambda k: ctypes.c_void_p(0x100000 * k)
    wts = PrologWeights(wq_a=0x1100000, gamma_cq=0x1200000, wq_b=0x1300000, w_uk=0x1400000, wkv=0x1500000,
                        gamma_ckv=0x1600000)
    args = [P(1), None, P(2), P(3), P(4), P(5), P(6), P(7), P(8), P(9), P(10)]  # x w cos sin idx qn qr kvn kvr sc ws
    ws_bytes = lib.mla_prolog_workspace_bytes(ctypes.byref(d))
    assert ws_bytes > 0
    dref = ctypes.byref(d)
    if case == "null_dims":
        dref = None
    elif case == "hidden_7":
        d.hidden = 7
    elif case == "q_lora_0":
        d.q_lora = 0
    elif case == "heads_0":
        d.n_heads = 0
    elif case == "eps_0":
        d.eps = 0.0
    elif case == "rows_0":
        d.num_rows = 0
    elif case == "int8_2":
        d.kv_int8 = 2
    elif case == "null_x":
        args[0] = None
    elif case == "null_weight":
        wts.w_uk = None
    elif case == "int8_no_scales":
        args[9] = None
    elif case == "misaligned_x":
        args[0] = ctypes.c_void_p(0x100008)
    elif case == "misaligned_gamma":
        wts.gamma_ckv = 0x1600002
    elif case == "misaligned_ws":
        args[10] = ctypes.c_void_p(0xA00080)
    elif case == "small_ws":
        ws_bytes -= 1
    elif case == "empty":
        d.T = 0
        args = [None] * 11
    st = lib.mla_prolog(dref, args[0], ctypes.byref(wts), *args[2:10], args[10], ctypes.c_size_t(ws_bytes), None)
    assert st == expect, (case, st, lib.mla_prolog_last_error())
    if expect != 0:
        assert lib.mla_prolog_last_error()


def test_debug_switch_reads_the_environment(monkeypatch):
    from mla_sparse_top_gb300 import binding
    monkeypatch.delenv("MLA_SPARSE_DEBUG", raising=False)
    assert not binding.debug_enabled()
    monkeypatch.setenv("MLA_SPARSE_DEBUG", "0")
    assert not binding.debug_enabled()
    monkeypatch.setenv("MLA_SPARSE_DEBUG", "1")
    assert binding.debug_enabled()
