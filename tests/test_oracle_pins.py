"""Pins for the fp64 oracle, independent of the oracle's own code.

Each check compares the oracle against something the pages or the mathematics
fix on their own: textbook dense attention over the un-paged cache restricted
to the selected positions (brute force), closed forms, invariances of the
definition, exact special values of the INT8 dequantisation rule, and the
flash online-softmax recurrence of the prefill section.  A plausible slip in
the oracle (a dropped rope term, a wrong block index, the value taken from the
wrong rows, the scale applied twice, the dequant rounding skipped) breaks at
least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Independent numpy round-to-nearest-even fp32 -> bf16 (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def numpy_dequant_bits(q8, scales):
    rows, d = q8.shape
    s = np.repeat(np.asarray(scales, np.float32), 128, axis=1)
    prod = q8.astype(np.float32) * s  # one fp32 multiply per element
    return f32_to_bf16_bits(prod)


def dense_cache_rows(inp, b):
    """Un-page batch b: logical position p -> physical row, for p < act."""
    bt = inp["block_table"][b]
    act = int(inp["act_seqs"][b])
    pos = np.arange(act)
    return bt[pos // 128].astype(np.int64) * 128 + pos % 128


def brute_force(inp, weights_per_token=None):
    """Textbook dense attention over all positions < act, with -inf outside the
    selected set (or a per-position multiplicity given explicitly)."""
    d = inp["dims"]
    T, H = d["B"] * d["S1"], d["n_q"]
    if d["kv_int8"]:
        kn_all = bf16_to_f64(numpy_dequant_bits(inp["kv_nope"], inp["kv_scales"]))
    else:
        kn_all = bf16_to_f64(inp["kv_nope"])
    kr_all = bf16_to_f64(inp["kv_rope"])
    out = np.zeros((T, H, d["d_nope"]))
    lse = np.full((T, H), -np.inf)
    for t in range(T):
        b = t // d["S1"]
        rows = dense_cache_rows(inp, b)
        act = rows.shape[0]
        if weights_per_token is None:
            w = np.zeros(act)
            sel = inp["topk_idx"][t]
            sel = sel[(sel >= 0) & (sel < act)]
            w[sel] = 1.0
        else:
            w = weights_per_token[t]
        if act == 0 or w.sum() == 0:
            continue
        K = np.concatenate([kn_all[rows], kr_all[rows]], axis=1)  # (act, 576)
        Q = np.concatenate([bf16_to_f64(inp["q_nope"][t]), bf16_to_f64(inp["q_rope"][t])], axis=1)  # (H, 576)
        S = inp["softmax_scale"] * (Q @ K.T)  # (H, act)
        logw = np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf)
        Z = S + logw[None, :]
        m = Z.max(axis=1, keepdims=True)
        E = np.exp(Z - m)
        l = E.sum(axis=1, keepdims=True)
        out[t] = (E @ kn_all[rows]) / l
        lse[t] = (m + np.log(l))[:, 0]
    return out, lse


def small(**kw):
    base = dict(B=2, S1=2, n_q=4, act_seqs=[300, 77], topk=50, seed=11, num_blocks=6)
    base.update(kw)
    return workloads.make_inputs(**base)


def test_oracle_builds_and_runs():
    inp = small()
    out, lse, bad = oracle.forward(inp)
    assert out.shape == (4, 4, 512) and lse.shape == (4, 4) and bad == 0
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("kv_int8", [False, True])
def test_matches_bruteforce_dense_masked(kv_int8):
    inp = small(kv_int8=kv_int8, act_seqs=[300, 130], topk=96)
    out, lse, _ = oracle.forward(inp)
    ref_out, ref_lse = brute_force(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_nondefault_softmax_scale_bruteforce():
    inp = small(topk=64, softmax_scale=0.3)
    out, lse, _ = oracle.forward(inp)
    ref_out, ref_lse = brute_force(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_pages_edge_lengths_bruteforce():
    """act_seq 16381 (not a multiple of 128) and 15 < topk, from the pages' case table."""
    cases = json.load(open(os.path.join(GOLDEN, "pages_test_cases.json")))
    acts = cases["cases"][0]["act_seqs"]  # [65536, 16381, 666, 15]
    inp = workloads.make_inputs(B=4, S1=1, n_q=2, act_seqs=[4096] + acts[1:], topk=cases["default_topk"], seed=5,
                                kv_int8=True)
    assert inp["act_seqs"][1] == 16381 and inp["act_seqs"][3] == 15
    out, lse, _ = oracle.forward(inp)
    ref_out, ref_lse = brute_force(inp)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    # act 15: all 15 positions selected, the remaining 2033 entries are -1
    assert (inp["topk_idx"][3] >= 0).sum() == 15


def test_single_valid_entry_closed_form():
    inp = small(topk=20)
    inp["topk_idx"][:] = -1
    inp["topk_idx"][0, 7] = 123  # batch 0 (act 300)
    out, lse, _ = oracle.forward(inp)
    r = dense_cache_rows(inp, 0)[123]
    kn = bf16_to_f64(inp["kv_nope"][r])
    kr = bf16_to_f64(inp["kv_rope"][r])
    z = inp["softmax_scale"] * (bf16_to_f64(inp["q_nope"][0]) @ kn + bf16_to_f64(inp["q_rope"][0]) @ kr)
    np.testing.assert_array_equal(out[0], np.broadcast_to(kn, out[0].shape))
    np.testing.assert_allclose(lse[0], z, rtol=1e-14, atol=1e-14)
    # tokens with nothing selected
    assert (out[1:] == 0).all() and np.isneginf(lse[1:]).all()


def test_zero_query_gives_mean_and_log_count():
    inp = small(topk=33)
    inp["q_nope"][:] = 0
    inp["q_rope"][:] = 0
    out, lse, _ = oracle.forward(inp)
    kn_all = bf16_to_f64(inp["kv_nope"])
    for t in range(4):
        b = t // 2
        sel = inp["topk_idx"][t]
        sel = sel[(sel >= 0) & (sel < inp["act_seqs"][b])]
        rows = dense_cache_rows(inp, b)[sel]
        np.testing.assert_allclose(out[t], np.broadcast_to(kn_all[rows].mean(0), out[t].shape), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[t], math.log(len(sel)), rtol=1e-14)


def test_identical_keys_give_that_row():
    inp = small(topk=40)
    rows = dense_cache_rows(inp, 1)
    inp["kv_nope"][rows] = inp["kv_nope"][rows[0]]
    inp["kv_rope"][rows] = inp["kv_rope"][rows[0]]
    out, lse, _ = oracle.forward(inp)
    kn = bf16_to_f64(inp["kv_nope"][rows[0]])
    kr = bf16_to_f64(inp["kv_rope"][rows[0]])
    for t in (2, 3):
        n = int(((inp["topk_idx"][t] >= 0) & (inp["topk_idx"][t] < 77)).sum())
        z = inp["softmax_scale"] * (bf16_to_f64(inp["q_nope"][t]) @ kn + bf16_to_f64(inp["q_rope"][t]) @ kr)
        np.testing.assert_allclose(out[t], np.broadcast_to(kn, out[t].shape), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[t], z + math.log(n), rtol=1e-13, atol=1e-13)


def test_rows_of_p_sum_to_one_via_constant_value():
    """With every selected value row equal to all-ones, out = sum_i p_i = 1."""
    inp = small(topk=64)
    inp["kv_nope"][:] = 0x3F80  # bf16 1.0 everywhere (keys differ only in rope)
    out, _, _ = oracle.forward(inp)
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)


def test_topk_permutation_and_padding_invariance():
    inp = small(topk=50)
    out0, lse0, _ = oracle.forward(inp)
    rng = np.random.default_rng(3)
    perm_inp = dict(inp)
    T = inp["topk_idx"].shape[0]
    wide = np.full((T, 80), -1, dtype=np.int32)
    for t in range(T):
        row = inp["topk_idx"][t]
        slots = np.sort(rng.choice(80, size=50, replace=False))
        wide[t, slots] = rng.permutation(row)
    perm_inp["topk_idx"] = wide
    perm_inp["dims"] = dict(inp["dims"], topk=80)
    out1, lse1, _ = oracle.forward(perm_inp)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13, atol=1e-13)


def test_physical_block_permutation_invariance():
    inp = small(topk=60, num_blocks=9)
    out0, lse0, _ = oracle.forward(inp)
    nb = inp["dims"]["num_blocks"]
    perm = np.random.default_rng(5).permutation(nb)  # new physical id of old block k is perm[k]
    moved = dict(inp)
    for key in ("kv_nope", "kv_rope"):
        src = inp[key].reshape(nb, 128, -1)
        dst = np.empty_like(src)
        dst[perm] = src
        moved[key] = dst.reshape(inp[key].shape)
    bt = inp["block_table"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved["block_table"] = bt
    out1, lse1, _ = oracle.forward(moved)
    np.testing.assert_array_equal(out1, out0)
    np.testing.assert_array_equal(lse1, lse0)


def test_nan_poisoned_unreferenced_rows_do_not_leak():
    inp = small(topk=50, num_blocks=8)  # 8 blocks, only 4 used; partial blocks beyond act poisoned too
    kn = inp["kv_nope"]
    assert (kn == workloads.BF16_NAN_BITS).any()
    out0, lse0, _ = oracle.forward(inp)
    assert np.isfinite(out0).all() and np.isfinite(lse0).all()
    clean = dict(inp)
    clean["kv_nope"] = np.where(kn == workloads.BF16_NAN_BITS, np.uint16(0x3F80), kn)
    out1, lse1, _ = oracle.forward(clean)
    np.testing.assert_array_equal(out1, out0)
    np.testing.assert_array_equal(lse1, lse0)


def test_int8_path_equals_bf16_path_on_dequantised_cache():
    inp = small(kv_int8=True, topk=64, poison_unused=False)
    deq = numpy_dequant_bits(inp["kv_nope"], inp["kv_scales"])
    np.testing.assert_array_equal(oracle.dequant_rows(inp["kv_nope"], inp["kv_scales"]), deq)
    out8, lse8, _ = oracle.forward(inp)
    bf = dict(inp)
    bf["kv_nope"] = deq
    bf["kv_scales"] = None
    bf["dims"] = dict(inp["dims"], kv_int8=0)
    outb, lseb, _ = oracle.forward(bf)
    np.testing.assert_array_equal(out8, outb)
    np.testing.assert_array_equal(lse8, lseb)


def test_dequant_exact_special_values():
    q = np.array([[127, -127, 1, -1, 0, -128] + [0] * 122], dtype=np.int8)
    for k in (0, 3, 7, 20):
        sc = np.array([[2.0 ** -k]], dtype=np.float32)
        got = bf16_to_f64(oracle.dequant_rows(q, sc))[0, :6]
        np.testing.assert_array_equal(got, np.array([127, -127, 1, -1, 0, -128]) * 2.0 ** -k)


def test_dequant_rounds_the_fp32_product_to_bf16():
    """A product that needs more than 8 significant bits is rounded to nearest-even bf16."""
    q = np.zeros((1, 128), dtype=np.int8)
    q[0, 0] = 3
    q[0, 1] = 101
    sc = np.array([[1.0 + 2.0 ** -8]], dtype=np.float32)  # 3 * (1 + 2^-8) needs 10 bits
    got = bf16_to_f64(oracle.dequant_rows(q, sc))[0, :2]
    exact = np.array([3, 101], dtype=np.float64) * (1.0 + 2.0 ** -8)
    assert got[0] != exact[0] and abs(got[0] - exact[0]) <= 2.0 ** -7 * 2  # half an ulp of 3.x in bf16
    np.testing.assert_array_equal(got, bf16_to_f64(f32_to_bf16_bits(np.float32(exact))))


def test_duplicate_indices_count_as_multiset():
    inp = small(topk=30)
    inp["topk_idx"][0, 1] = inp["topk_idx"][0, 0]  # entry 0 now appears twice
    out, lse, _ = oracle.forward(inp)
    T = 4
    weights = []
    for t in range(T):
        b = t // 2
        act = int(inp["act_seqs"][b])
        w = np.zeros(act)
        for j in inp["topk_idx"][t]:
            if 0 <= j < act:
                w[j] += 1.0
        weights.append(w)
    ref_out, ref_lse = brute_force(inp, weights_per_token=weights)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_flash_online_softmax_recurrence_equals_direct():
    """The prefill section's update (m_new = max(m, m~), l and o rescaled by
    exp(m - m_new), normalised only after the last tile) over 64-key tiles gives
    the decode-mode result."""
    inp = small(topk=200, act_seqs=[300, 250], n_q=3)
    out, lse, _ = oracle.forward(inp)
    kn_all = bf16_to_f64(inp["kv_nope"])
    kr_all = bf16_to_f64(inp["kv_rope"])
    for t in range(4):
        b = t // 2
        sel = inp["topk_idx"][t]
        sel = sel[(sel >= 0) & (sel < inp["act_seqs"][b])]
        rows = dense_cache_rows(inp, b)[sel]
        Q = np.concatenate([bf16_to_f64(inp["q_nope"][t]), bf16_to_f64(inp["q_rope"][t])], axis=1)
        m = np.full(Q.shape[0], -np.inf)
        l = np.zeros(Q.shape[0])
        o = np.zeros((Q.shape[0], 512))
        for j0 in range(0, len(rows), 64):
            r = rows[j0:j0 + 64]
            S = inp["softmax_scale"] * (Q @ np.concatenate([kn_all[r], kr_all[r]], axis=1).T)
            mt = S.max(axis=1)
            P = np.exp(S - mt[:, None])
            lt = P.sum(axis=1)
            m_new = np.maximum(m, mt)
            a, c = np.exp(m - m_new), np.exp(mt - m_new)
            l = a * l + c * lt
            o = a[:, None] * o + c[:, None] * (P @ kn_all[r])
            m = m_new
        np.testing.assert_allclose(out[t], o / l[:, None], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[t], m + np.log(l), rtol=1e-12)


def test_bad_block_ids_are_masked_and_counted():
    inp = small(topk=50)
    bt = inp["block_table"].copy()
    victim = bt[0, 0]
    inp2 = dict(inp)
    bt[0, 0] = 999  # out of range for valid positions 0..127 of batch 0
    inp2["block_table"] = bt
    out, lse, bad = oracle.forward(inp2)
    sel = inp["topk_idx"][:2]
    expect_bad = int(((sel >= 0) & (sel < 128)).sum())
    assert bad == expect_bad > 0
    # same as dropping those entries from the list
    inp3 = dict(inp)
    tk = inp["topk_idx"].copy()
    tk[:2][(tk[:2] >= 0) & (tk[:2] < 128)] = -1
    inp3["topk_idx"] = tk
    out3, lse3, _ = oracle.forward(inp3)
    np.testing.assert_array_equal(out[:2], out3[:2])
    assert victim >= 0


def test_tiny_decode_matches_stored_oracle_values():
    """Regression fixture written by tests/golden/make_oracle_fixture.py (oracle only)."""
    fx = json.load(open(os.path.join(GOLDEN, "tiny_decode_oracle.json")))
    inp = workloads.tiny_decode(seed=fx["seed"])
    out, lse, _ = oracle.forward(inp)
    for (h, dd), v in zip(fx["out_index"], fx["out_values"]):
        assert out[0, h, dd] == pytest.approx(v, rel=1e-12, abs=1e-15)
    np.testing.assert_allclose(lse[0], fx["lse"], rtol=1e-12)
