"""Pins of the Lightning Indexer oracle ("CANN DeepSeek Indexer attention",
sections "Lightning Indexer" and "Sparse Flash Attention"): independent numpy
brute force on an un-paged cache, closed forms, the selection rule checked
against a plain sort, and invariants.  CPU only."""
import numpy as np
import pytest

import oracle
import workloads


def bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round-to-nearest-even fp64 -> bf16 bits (test-side helper for building inputs)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def dense_cache(inp, b):
    """The logical key rows 0..act-1 of sequence b, un-paged with the table (independent of the oracle)."""
    d = inp["dims"]
    act = int(inp["act_seqs"][b])
    rows = []
    for j in range(act):
        blk = inp["block_table"][b, j // d["block_size"]]
        rows.append(inp["k_cache"][blk * d["block_size"] + j % d["block_size"]])
    return bf16_f64(np.array(rows, dtype=np.uint16).reshape(act, d["head_dim"]))


def brute_scores(inp):
    d = inp["dims"]
    T = d["B"] * d["S1"]
    out = []
    for t in range(T):
        b = t // d["S1"]
        k = dense_cache(inp, b)                               # (act, D)
        q = bf16_f64(inp["q"][t])                             # (H, D)
        dots = np.einsum("hd,jd->hj", q, k)                   # (H, act)
        out.append(np.einsum("h,hj->j", inp["w"][t].astype(np.float64), np.maximum(dots, 0.0)))
    return out


def plain_select(scores_row, act, k):
    s = np.asarray(scores_row[:act], dtype=np.float64)
    cand = np.nonzero(s != -np.inf)[0]
    order = np.lexsort((cand, -s[cand]))                      # score descending, position ascending
    chosen = np.sort(cand[order[:k]])
    res = np.full(k, -1, dtype=np.int32)
    res[: len(chosen)] = chosen
    return res


@pytest.mark.parametrize("maker", [workloads.indexer_tiny,
                                   lambda: workloads.make_indexer_inputs(B=2, S1=2, n_heads=4, act_seqs=[200, 331],
                                                                         topk=50, seed=11, num_blocks=7)])
def test_scores_equal_dense_brute_force(maker):
    inp = maker()
    sc, bad = oracle.indexer_scores(inp)
    assert bad == 0
    ref = brute_scores(inp)
    d = inp["dims"]
    for t in range(d["B"] * d["S1"]):
        act = int(inp["act_seqs"][t // d["S1"]])
        np.testing.assert_allclose(sc[t, :act], ref[t], rtol=1e-12, atol=1e-9)
        assert np.all(sc[t, act:] == -np.inf)


def test_selection_equals_plain_sort():
    inp = workloads.make_indexer_inputs(B=3, S1=2, n_heads=4, act_seqs=[500, 129, 40], topk=64, seed=12)
    sc, _ = oracle.indexer_scores(inp)
    sel = oracle.indexer_select(sc, inp["act_seqs"], 2, 64)
    for t in range(6):
        np.testing.assert_array_equal(sel[t], plain_select(sc[t], int(inp["act_seqs"][t // 2]), 64))
    # fewer candidates than k: all positions, then -1
    np.testing.assert_array_equal(sel[4, :40], np.arange(40))
    assert np.all(sel[4, 40:] == -1)


def test_zero_weights_select_the_first_positions():
    inp = workloads.make_indexer_inputs(B=1, S1=1, n_heads=4, act_seqs=[300], topk=32, seed=13, w_scale=0.0)
    sc, _ = oracle.indexer_scores(inp)
    assert np.all(sc[0, :300] == 0.0)
    np.testing.assert_array_equal(oracle.indexer_select(sc, inp["act_seqs"], 1, 32)[0], np.arange(32))


def test_closed_form_single_head_query_equal_to_a_key():
    inp = workloads.make_indexer_inputs(B=1, S1=1, n_heads=1, act_seqs=[256], topk=1, seed=14)
    k = dense_cache(inp, 0)
    j0 = 77
    inp["q"][0, 0] = f64_to_bf16_bits(k[j0])                  # q = k_j0 exactly (bf16 values)
    inp["w"][0, 0] = 1.0
    sc, _ = oracle.indexer_scores(inp)
    assert sc[0, j0] == pytest.approx(float(np.dot(k[j0], k[j0])), rel=1e-15)
    # Cauchy-Schwarz makes j0 the unique maximiser unless another row is parallel and longer
    best = int(np.argmax(sc[0, :256]))
    assert sc[0, best] >= sc[0, j0]
    assert oracle.indexer_select(sc, inp["act_seqs"], 1, 1)[0, 0] == best


def test_relu_drops_negative_dots():
    inp = workloads.make_indexer_inputs(B=1, S1=1, n_heads=1, act_seqs=[128], topk=4, seed=15)
    k = dense_cache(inp, 0)
    inp["q"][0, 0] = f64_to_bf16_bits(-k[5])
    inp["w"][0, 0] = 2.0
    sc, _ = oracle.indexer_scores(inp)
    assert sc[0, 5] == 0.0
    dots = k @ bf16_f64(inp["q"][0, 0])
    np.testing.assert_allclose(sc[0, :128], 2.0 * np.maximum(dots, 0.0), rtol=1e-12, atol=1e-12)


def test_ties_at_the_threshold_go_to_the_smaller_position():
    inp = workloads.make_indexer_inputs(B=1, S1=1, n_heads=2, act_seqs=[256], topk=10, seed=16)
    sc, _ = oracle.indexer_scores(inp)
    s = sc[0].copy()
    order = np.argsort(-s[:256], kind="stable")
    thr_pos = order[9]                                        # the 10th best
    later = [j for j in range(256) if j > thr_pos and s[j] < s[thr_pos]][0]
    earlier = [j for j in range(256) if j < thr_pos and s[j] < s[thr_pos]][0]
    s[later] = s[thr_pos]                                     # a tie with a larger position: loses
    sel = oracle.indexer_select(s[None, :], inp["act_seqs"], 1, 10)[0]
    assert thr_pos in sel and later not in sel
    s[earlier] = s[thr_pos]                                   # a tie with a smaller position: wins over thr_pos
    sel = oracle.indexer_select(s[None, :], inp["act_seqs"], 1, 10)[0]
    assert earlier in sel and thr_pos not in sel


def test_block_permutation_and_positive_weight_scale_invariance():
    inp = workloads.make_indexer_inputs(B=2, S1=2, n_heads=4, act_seqs=[384, 300], topk=40, seed=17,
                                        poison_unused=False)
    sc, _ = oracle.indexer_scores(inp)
    sel = oracle.indexer_select(sc, inp["act_seqs"], 2, 40)
    # physical blocks permuted, table rewritten
    d = inp["dims"]
    nb = d["num_blocks"]
    perm = np.random.default_rng(0).permutation(nb)
    cache2 = np.empty_like(inp["k_cache"])
    for old in range(nb):
        cache2[perm[old] * 128:(perm[old] + 1) * 128] = inp["k_cache"][old * 128:(old + 1) * 128]
    inp2 = dict(inp, k_cache=cache2, block_table=np.where(inp["block_table"] >= 0, perm[inp["block_table"]], -1)
                .astype(np.int32))
    sc2, _ = oracle.indexer_scores(inp2)
    np.testing.assert_array_equal(sc, sc2)
    # w scaled by 4 (exact in binary): scores scale, the selection does not move
    inp3 = dict(inp, w=inp["w"] * np.float32(4.0))
    sc3, _ = oracle.indexer_scores(inp3)
    np.testing.assert_array_equal(oracle.indexer_select(sc3, inp["act_seqs"], 2, 40), sel)


def test_bad_blocks_are_not_candidates():
    inp = workloads.make_indexer_inputs(B=1, S1=1, n_heads=2, act_seqs=[256], topk=200, seed=18)
    inp["block_table"][0, 1] = 9999                           # positions 128..255 lose their block
    sc, bad = oracle.indexer_scores(inp)
    assert bad == 128
    assert np.all(sc[0, 128:256] == -np.inf)
    sel = oracle.indexer_select(sc, inp["act_seqs"], 1, 200)[0]
    np.testing.assert_array_equal(sel[:128], np.arange(128))
    assert np.all(sel[128:] == -1)
