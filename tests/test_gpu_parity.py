"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Small cases are compared element by element in full; the full-size workloads
(the launch configuration the benchmark times) are compared on sampled tokens
that the oracle evaluates one by one.  Tolerance: rtol 5e-3 / atol 1e-4 on the
bf16 output, 1e-3 relative on lse.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import assert_lse_close, assert_out_close, run_gpu, to_device, launch  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_sparse_top_gb300 import build
    build.build()


def check_full(inp, label, mode=None):
    out, lse, status = run_gpu(inp, mode=mode)
    ref_out, ref_lse, bad = oracle.forward(inp)
    assert status == (1 if bad else 0), f"{label}: device status {status:#x}"
    assert_out_close(out, ref_out, label)
    assert_lse_close(lse, ref_lse, label)
    return out, lse


def check_sampled(inp, label, n_sample=8, seed=0, tokens=None):
    T = inp["dims"]["B"] * inp["dims"]["S1"]
    if tokens is None:
        rng = np.random.default_rng(seed)
        toks = sorted(set([0, T - 1] + rng.choice(T, size=min(T, n_sample), replace=False).tolist()))
    else:
        toks = sorted(set(int(t) for t in tokens))
    out, lse, status = run_gpu(inp)
    ref_out, ref_lse, bad = oracle.forward(inp, tokens=toks)
    assert status & 2 == 0, f"{label}: device timeout"
    assert_out_close(out[toks], ref_out, label)
    assert_lse_close(lse[toks], ref_lse, label)
    assert np.isfinite(out).all()


def test_tiny_decode_full():
    check_full(workloads.tiny_decode(), "tiny_decode")


@pytest.mark.parametrize("kv_int8", [False, True])
def test_ragged_multi_tile(kv_int8):
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[1000, 300], topk=200, seed=21, num_blocks=12,
                                kv_int8=kv_int8)
    check_full(inp, f"ragged int8={kv_int8}")


def test_mtp_decode_reduced_batch():
    check_full(workloads.mtp_decode(B=3), "mtp_decode B=3")


def test_int8_decode_reduced_batch():
    check_full(workloads.int8_decode(B=3), "int8_decode B=3")


def test_pages_case_total_int8_exact_shape():
    """B=4 S1=2 N_Q=128 act [65536, 16381, 666, 15] INT8, topk 2048 (the pages' first case)."""
    case = json.load(open(os.path.join(GOLDEN, "pages_test_cases.json")))["cases"][0]
    inp = workloads.make_inputs(B=case["B"], S1=case["S1"], n_q=case["N_Q"], act_seqs=case["act_seqs"], topk=2048,
                                seed=31, kv_int8=True)
    check_full(inp, case["name"])


@pytest.mark.parametrize("ci", [1, 2, 4])
def test_pages_cases_64k(ci):
    case = json.load(open(os.path.join(GOLDEN, "pages_test_cases.json")))["cases"][ci]
    inp = workloads.make_inputs(B=case["B"], S1=case["S1"], n_q=case["N_Q"], act_seqs=case["act_seqs"], topk=2048,
                                seed=40 + ci, kv_int8=case["kv"] == "int8")
    check_full(inp, case["name"])


def test_pages_case_prefill_256_sampled():
    case = json.load(open(os.path.join(GOLDEN, "pages_test_cases.json")))["cases"][3]
    act = case["act_seqs"][0]
    pos = np.arange(act - case["S1"], act).reshape(1, -1)
    inp = workloads.make_inputs(B=1, S1=case["S1"], n_q=128, act_seqs=[act], topk=2048, seed=43, kv_int8=True,
                                positions=pos, mode="prefill")
    check_sampled(inp, case["name"], n_sample=12)


def test_varlen_reduced():
    inp = workloads.make_inputs(B=6, S1=2, n_q=128, act_seqs=[65536, 16381, 666, 15, 2048, 2047], topk=2048, seed=23)
    check_full(inp, "varlen B=6")


def test_prefill_reduced_and_mode_equivalence():
    act = 4096
    pos = np.arange(act - 48, act).reshape(1, -1)
    inp = workloads.make_inputs(B=1, S1=48, n_q=128, act_seqs=[act], topk=2048, seed=24, positions=pos,
                                mode="prefill")
    out_p, lse_p = check_full(inp, "prefill S1=48", mode="prefill")
    out_d, lse_d, _ = run_gpu(inp, mode="decode")
    np.testing.assert_array_equal(out_d, out_p)
    np.testing.assert_array_equal(lse_d, lse_p)


def test_early_prefill_positions_fewer_than_topk():
    pos = np.arange(0, 40).reshape(1, -1) * 37  # positions 0..1443: candidates p+1 < 2048
    inp = workloads.make_inputs(B=1, S1=40, n_q=128, act_seqs=[1500], topk=2048, seed=25, positions=pos,
                                mode="prefill")
    check_full(inp, "early prefill")


@pytest.mark.parametrize("kv_int8", [False, True])
@pytest.mark.parametrize("n_q", [1, 16, 50, 100])
def test_head_counts(n_q, kv_int8):
    # head counts that end inside a group of four lanes: Q and out move line-major
    # through four-lane transposes that mix live and absent heads
    inp = workloads.make_inputs(B=2, S1=1, n_q=n_q, act_seqs=[777, 129], topk=130, seed=26, num_blocks=10,
                                kv_int8=kv_int8)
    check_full(inp, f"n_q={n_q} int8={kv_int8}")


def test_topk_one_and_tiny_lists():
    for topk in (1, 63, 64, 65):
        inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[500, 70], topk=topk, seed=27 + topk)
        check_full(inp, f"topk={topk}")


def test_all_masked_and_empty_sequences():
    inp = workloads.make_inputs(B=3, S1=2, n_q=128, act_seqs=[300, 0, 200], topk=96, seed=28, num_blocks=6)
    inp["topk_idx"][0] = -1  # token 0: nothing selected
    inp["topk_idx"][5, :] = 5000  # token 5: only out-of-range indices
    out, lse = check_full(inp, "masked")
    for t in (0, 2, 3, 5):
        assert (out[t] == 0).all() and np.isneginf(lse[t]).all()


def test_duplicate_indices():
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[600, 600], topk=150, seed=29)
    inp["topk_idx"][:, 100:150] = inp["topk_idx"][:, :50]
    check_full(inp, "duplicates")


def test_bad_block_ids_are_masked_and_flagged():
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[600, 300], topk=150, seed=30)
    inp["block_table"][0, 1] = 10 ** 6
    out, lse, status = run_gpu(inp)
    ref_out, ref_lse, bad = oracle.forward(inp)
    assert bad > 0 and status == 1
    assert_out_close(out, ref_out, "bad blocks")
    assert_lse_close(lse, ref_lse, "bad blocks")


def test_large_logits_trigger_rescale():
    """Queries scaled so that scores span a wide range: exercises the running-max rescale of O."""
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[3000, 3000], topk=1024, seed=32)
    q = inp["q_nope"].astype(np.int32)
    nz = (q & 0x7FFF) != 0
    inp["q_nope"] = np.where(nz, q + (4 << 7), q).astype(np.uint16)  # x16, exact in bf16
    check_full(inp, "large logits")


def test_softmax_scale_variants():
    """Positive scales take the row max on raw scores; zero and negative
    scales scale every score before the max (the other branch)."""
    for scale in (0.01, 0.3, 0.0, -0.05, -1.0):
        inp = workloads.make_inputs(B=1, S1=2, n_q=128, act_seqs=[900], topk=256, seed=33, softmax_scale=scale)
        check_full(inp, f"scale={scale}")


def test_deterministic_and_permutation_stable():
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[2500, 2500], topk=512, seed=34)
    dev = to_device(inp)
    a = run_gpu(inp, dev=dev)
    b = run_gpu(inp, dev=dev)
    np.testing.assert_array_equal(a[0], b[0])
    perm = inp.copy()
    perm["topk_idx"] = inp["topk_idx"][:, np.random.default_rng(0).permutation(512)].copy()
    c = run_gpu(perm)
    ref_out, ref_lse, _ = oracle.forward(inp)
    assert_out_close(c[0], ref_out, "permuted list")


# ------------------------------------------------------------ full-size workloads
# The launch configuration the benchmark times.  The 128-token decode
# workloads are checked on every token; the 4096-token prefill on 274 tokens,
# every 15th one plus the last (15 is prime to the number of clusters, so the
# sample covers every cluster and many stream positions).
@pytest.mark.parametrize("name", ["mtp_decode", "int8_decode", "varlen_decode", "mtp_decode_b2"])
def test_full_size_decode_every_token(name):
    inp = workloads.NAMED[name]()
    T = inp["dims"]["B"] * inp["dims"]["S1"]
    check_sampled(inp, name, tokens=range(T))


def test_full_size_prefill_strided_tokens():
    inp = workloads.NAMED["prefill"]()
    T = inp["dims"]["B"] * inp["dims"]["S1"]
    toks = list(range(0, T, 15)) + [T - 1]
    assert len(set(toks)) >= 256 and 0 in toks and T - 1 in toks
    check_sampled(inp, "prefill", tokens=toks)


# ------------------------------------------------------------ persistent clusters: token streams
# The kernel runs at most as many two-CTA clusters as the GPU holds at once
# (76 on GB300); cluster c takes tokens c, c + G, ... as one stream of key
# tiles.  These cases move the token boundaries through the stream.
@pytest.mark.parametrize("kv_int8", [False, True])
def test_one_tile_per_token_long_streams(kv_int8):
    """topk = 64: every tile is a token boundary (Q reload, O hand-off and the
    row-sum handshake on every tile); 1200 tokens, ~16 per cluster."""
    B, S1 = 600, 2
    act = np.random.default_rng(40).integers(1, 400, size=B)
    inp = workloads.make_inputs(B=B, S1=S1, n_q=128, act_seqs=act, topk=64, seed=40, kv_int8=kv_int8)
    check_full(inp, f"one tile per token int8={kv_int8}")


@pytest.mark.parametrize("B", [38, 39, 77])
def test_token_counts_around_the_cluster_count(B):
    """T = 76, 78 and 154 tokens: one token per cluster, two clusters with a
    second token, and every cluster with two or three; topk 100 leaves a
    partial last tile in every token."""
    inp = workloads.make_inputs(B=B, S1=2, n_q=128, act_seqs=[700] * B, topk=100, seed=41 + B)
    check_full(inp, f"T={2 * B}")


def test_rescale_inside_a_later_token_of_the_stream():
    """Large logits in tokens that are a cluster's second or third: the O
    rescale must act on the accumulator of the current token only."""
    B = 100
    inp = workloads.make_inputs(B=B, S1=2, n_q=64, act_seqs=[600] * B, topk=192, seed=45)
    q = inp["q_nope"].astype(np.int32)
    nz = (q & 0x7FFF) != 0
    scaled = np.where(nz, q + (4 << 7), q).astype(np.uint16)  # x16, exact in bf16
    inp["q_nope"][160:] = scaled[160:]
    check_full(inp, "rescale in later tokens")


def test_output_aligned_to_16_bytes_only():
    """`out` only has to be 16-byte aligned: the epilogue then stores 16 bytes
    per instruction instead of 32.  Same bits either way, and the oracle's."""
    inp = workloads.make_inputs(B=3, S1=2, n_q=128, act_seqs=[3000, 700, 5000], topk=1000, seed=91)
    dev = to_device(inp)
    out32, lse32, status = run_gpu(inp, dev=dev)
    assert status == 0
    big = torch.empty(dev["out"].numel() + 8, dtype=dev["out"].dtype, device="cuda")
    dev["out"] = big[8:].view(dev["out"].shape)
    assert dev["out"].data_ptr() % 32 == 16
    out16, lse16, status = run_gpu(inp, dev=dev)
    assert status == 0
    np.testing.assert_array_equal(out16, out32)
    np.testing.assert_array_equal(lse16, lse32)
    ref_out, ref_lse, _ = oracle.forward(inp)
    assert_out_close(out16, ref_out, "out at a 16-byte offset")
    assert_lse_close(lse16, ref_lse, "out at a 16-byte offset")
