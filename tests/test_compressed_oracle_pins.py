"""Pins of the compressed / sparse compressed attention oracle (CFA / SCFA;
"NPU DeepSeek-V4 PyPTO fused-operator optimization", sections CFA, SCFA and
Compressor; readings in oracle/compressed.py), each against something other
than itself: the C window oracle, the C sparse-attention oracle on an
equivalent explicit list, the CFA form, permutations, and the C dequantiser.
CPU only."""
import numpy as np
import pytest

import oracle
import oracle.compressed as comp
import workloads


def small(**kw):
    base = dict(B=3, S1=2, n_q=8, act_seqs=[300, 41, 257], window=16, cmp_ratio=4, seed=120)
    base.update(kw)
    return workloads.make_compressed_inputs(**base)


def test_without_visible_compressed_entries_it_is_window_attention():
    inp = small(cmp_ratio=1000)                                           # no entry is complete yet
    out, lse, bad = comp.forward(inp, 16, 1000)
    ref_out, ref_lse, _ = oracle.swa_forward(inp, 16)
    assert bad == 0
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


@pytest.mark.parametrize("window,ratio", [(16, 4), (1, 8), (40, 128)])
def test_cfa_with_copied_rows_is_sparse_attention_over_the_same_positions(window, ratio):
    """Let compressed entry i hold a copy of the original row at position i*r:
    CFA must then equal sparse attention (the C oracle) over the window
    positions plus the positions i*r of the visible entries."""
    inp = small(window=window, cmp_ratio=ratio, act_seqs=[300, 41, 257])
    d = inp["dims"]
    for b in range(d["B"]):
        act = int(inp["act_seqs"][b])
        for i in range(act // ratio):
            src = inp["block_table"][b, (i * ratio) // 128] * 128 + (i * ratio) % 128
            dst = inp["cmp_block_table"][b, i // 128] * 128 + i % 128
            inp["cmp_nope"][dst] = inp["kv_nope"][src]
            inp["cmp_rope"][dst] = inp["kv_rope"][src]
    out, lse, bad = comp.forward(inp, window, ratio)
    assert bad == 0
    T, S1 = d["B"] * d["S1"], d["S1"]
    lists = []
    for t in range(T):
        b, s = divmod(t, S1)
        p = int(inp["act_seqs"][b]) - S1 + s
        lst = [j for j in range(max(0, p - window + 1), p + 1)]
        lst += [i * ratio for i in range(0, max(0, (p + 1) // ratio))]
        lists.append(lst)
    K = max(len(x) for x in lists)
    topk = np.full((T, K), -1, dtype=np.int32)
    for t, lst in enumerate(lists):
        topk[t, :len(lst)] = lst
    ref_out, ref_lse, _ = oracle.forward(dict(inp, topk_idx=topk, dims=dict(d, topk=K)))
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_scfa_listing_every_visible_entry_is_cfa():
    inp = small()
    d = inp["dims"]
    T = d["B"] * d["S1"]
    K = 300 // 4
    lists = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        b, s = divmod(t, d["S1"])
        p = int(inp["act_seqs"][b]) - d["S1"] + s
        vis = (p + 1) // 4
        lists[t, :vis] = np.arange(vis)[::-1]
    a = comp.forward(inp, 16, 4)
    b2 = comp.forward(inp, 16, 4, cmp_idx=lists)
    np.testing.assert_allclose(b2[0], a[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b2[1], a[1], rtol=1e-12)


def test_scfa_ignores_order_padding_and_invisible_entries():
    inp = small(cmp_topk=12)
    lists = inp["cmp_idx"]
    a = comp.forward(inp, 16, 4, cmp_idx=lists)
    rng = np.random.default_rng(0)
    shuffled = np.stack([row[rng.permutation(row.shape[0])] for row in lists])
    padded = np.concatenate([shuffled, np.full((lists.shape[0], 3), -1, np.int32),
                             np.full((lists.shape[0], 2), 10 ** 6, np.int32)], axis=1)  # never visible
    b2 = comp.forward(inp, 16, 4, cmp_idx=padded)
    np.testing.assert_allclose(b2[0], a[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b2[1], a[1], rtol=1e-12)


def test_int8_caches_equal_bf16_caches_holding_their_dequantised_rows():
    inp = small(kv_int8=True, cmp_topk=10)
    a = comp.forward(inp, 16, 4, cmp_idx=inp["cmp_idx"])
    bf = dict(inp, kv_nope=oracle.dequant_rows(inp["kv_nope"], inp["kv_scales"]),
              cmp_nope=oracle.dequant_rows(inp["cmp_nope"], inp["cmp_scales"]), kv_scales=None, cmp_scales=None,
              dims=dict(inp["dims"], kv_int8=0))
    b2 = comp.forward(bf, 16, 4, cmp_idx=inp["cmp_idx"])
    np.testing.assert_array_equal(a[0], b2[0])
    np.testing.assert_array_equal(a[1], b2[1])


def test_token_with_nothing_to_attend_gives_zero_and_minus_inf():
    inp = small(act_seqs=[1, 41, 257])                                    # token (0, 0) sits at position -1
    out, lse, _ = comp.forward(inp, 16, 4, tokens=[0, 1])
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()
