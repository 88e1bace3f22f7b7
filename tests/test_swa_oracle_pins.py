"""Pins of the sliding-window attention oracle ("NPU DeepSeek-V4 PyPTO
fused-operator optimization", section SWA; readings in oracle/swa_oracle.c):
a dense numpy brute force over each token's window, a window as long as the
sequence equals causal attention, a one-position window returns that row.
CPU only."""
import numpy as np
import pytest

import oracle
import workloads


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense_window_attention(inp, window):
    """Independent brute force: un-page each sequence, take positions
    max(0, p - window + 1) .. p of token (b, s) with p = act_b - S1 + s, and
    run textbook softmax attention (bf16 caches only)."""
    d = inp["dims"]
    S1, H = d["S1"], d["n_q"]
    kn_all, kr_all = bf16_to_f64(inp["kv_nope"]), bf16_to_f64(inp["kv_rope"])
    outs, lses = [], []
    for b in range(d["B"]):
        act = int(inp["act_seqs"][b])
        rows = inp["block_table"][b][np.arange(act) // 128].astype(np.int64) * 128 + np.arange(act) % 128
        for s in range(S1):
            t = b * S1 + s
            p = act - S1 + s
            pos = np.arange(max(0, p - window + 1), p + 1)
            qn, qr = bf16_to_f64(inp["q_nope"][t]), bf16_to_f64(inp["q_rope"][t])  # (H, 512), (H, 64)
            if pos.size == 0:
                outs.append(np.zeros((H, 512)))
                lses.append(np.full(H, -np.inf))
                continue
            kn, kr = kn_all[rows[pos]], kr_all[rows[pos]]
            z = (qn @ kn.T + qr @ kr.T) * inp["softmax_scale"]
            m = z.max(axis=1, keepdims=True)
            e = np.exp(z - m)
            outs.append((e @ kn) / e.sum(axis=1, keepdims=True))
            lses.append(m[:, 0] + np.log(e.sum(axis=1)))
    return np.array(outs), np.array(lses)


@pytest.mark.parametrize("window,S1", [(1, 1), (7, 2), (64, 2), (130, 3), (1000, 2)])
def test_window_attention_equals_dense_brute_force(window, S1):
    inp = workloads.make_inputs(B=3, S1=S1, n_q=8, act_seqs=[300, 5, 129], topk=16, seed=80 + window)
    out, lse, bad = oracle.swa_forward(inp, window)
    ref_out, ref_lse = dense_window_attention(inp, window)
    assert bad == 0
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_window_covering_the_sequence_is_causal_attention():
    inp = workloads.make_inputs(B=2, S1=4, n_q=4, act_seqs=[200, 90], topk=16, seed=90)
    a = oracle.swa_forward(inp, 200)
    b = oracle.swa_forward(inp, 5000)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    # the newest token of each sequence sees every position: its lse is the log-sum-exp over all of them
    ref_out, ref_lse = dense_window_attention(inp, 10 ** 6)
    np.testing.assert_allclose(a[1], ref_lse, rtol=1e-12)


def test_one_position_window_returns_that_row():
    inp = workloads.make_inputs(B=2, S1=2, n_q=4, act_seqs=[260, 3], topk=16, seed=91)
    out, lse, _ = oracle.swa_forward(inp, 1)
    kn_all = bf16_to_f64(inp["kv_nope"])
    for b in range(2):
        act = int(inp["act_seqs"][b])
        for s in range(2):
            p = act - 2 + s
            row = inp["block_table"][b][p // 128] * 128 + p % 128
            np.testing.assert_array_equal(out[b * 2 + s], np.broadcast_to(kn_all[row], (4, 512)))


def test_window_lists():
    lists = oracle.swa_window_lists([5, 2], 2, 4)
    np.testing.assert_array_equal(lists, [[0, 1, 2, 3], [1, 2, 3, 4], [-1, -1, -1, 0], [-1, -1, 0, 1]])
