"""Tokens whose key tiles are split between persistent clusters.

The clusters take equal shares of the (token, tile) stream, so a token's tiles
may be cut between two or more clusters; each part keeps its own online
softmax state (O relative to its running max, the row sum) and the part that
finishes last merges them with the flash update's weights ("DeepSeek V3/V2
Sparse Flash Attention with Quantization", section "Flash online softmax
incremental update").  These cases cut tokens in every way the schedule can:
one token over 32 clusters (one tile each), three tokens over all clusters,
many tokens with cuts at both ends of a cluster.  A first call on a stream
that is capturing a CUDA graph has no buffer for cut tokens and schedules
whole tokens; a graph captured after the buffer exists cuts tokens and must
give the same result on every replay (the arrival words are left clear).
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import assert_lse_close, assert_out_close, launch, run_gpu, to_device  # noqa: E402


def _check(inp, label):
    out, lse, status = run_gpu(inp)
    assert status == 0, f"{label}: device status {status:#x}"
    ref_out, ref_lse, _ = oracle.forward(inp)
    assert_out_close(out, ref_out, label)
    assert_lse_close(lse, ref_lse, label)


@pytest.mark.parametrize("B, S1, act, topk, seed", [
    (1, 1, 8192, 2048, 80),            # one token, 32 tiles: 32 clusters of one tile
    (3, 1, 6000, 2048, 81),            # 96 tiles over every cluster
    (5, 2, 3000, 1000, 82),            # ragged last tile, cuts at both ends of clusters
    (1, 2, 300, 2048, 83),             # mostly padded lists: parts with no valid key
])
def test_cut_tokens_match_the_oracle(B, S1, act, topk, seed):
    inp = workloads.make_inputs(B=B, S1=S1, n_q=128, act_seqs=[act] * B, topk=topk, seed=seed)
    _check(inp, f"B={B} S1={S1} act={act} topk={topk}")


def test_cut_tokens_int8_and_few_heads():
    inp = workloads.make_inputs(B=2, S1=1, n_q=48, act_seqs=[7000, 5000], topk=2048, seed=84, kv_int8=True)
    _check(inp, "int8 n_q=48")


def _to_np(dev):
    from gpu_util import bf16_to_f64
    out = bf16_to_f64(dev["out"].view(torch.int16).cpu().numpy().view(np.uint16))
    return out, dev["lse"].cpu().numpy().astype(np.float64)


def test_graph_capture_with_and_without_the_buffer():
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_inputs(B=3, S1=1, n_q=128, act_seqs=[6000, 4000, 8000], topk=2048, seed=85)
    ref_out, ref_lse, _ = oracle.forward(inp)
    dev = to_device(inp)
    run_gpu(inp, dev=dev)  # kernel set-up happens outside any capture
    assert mla.device_status(clear=True) == 0
    # a fresh stream: its first call is made under capture (whole tokens)
    side = torch.cuda.Stream()
    g0 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g0, stream=side):
        launch(inp, dev)
    for rep in range(2):
        dev["out"].fill_(float("nan"))
        g0.replay()
        torch.cuda.synchronize()
        out, lse = _to_np(dev)
        assert_out_close(out, ref_out, f"captured without a buffer, replay {rep}")
        assert_lse_close(lse, ref_lse, f"captured without a buffer, replay {rep}")
    # an ordinary call on that stream allocates the buffer; a graph captured
    # afterwards cuts tokens
    with torch.cuda.stream(side):
        dev["out"].fill_(float("nan"))
        launch(inp, dev)
    torch.cuda.synchronize()
    out, lse = _to_np(dev)
    assert_out_close(out, ref_out, "eager call on the side stream")
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=side):
        launch(inp, dev)
    for rep in range(3):
        dev["out"].fill_(float("nan"))
        g1.replay()
        torch.cuda.synchronize()
        out, lse = _to_np(dev)
        assert_out_close(out, ref_out, f"captured with the buffer, replay {rep}")
        assert_lse_close(lse, ref_lse, f"captured with the buffer, replay {rep}")
    assert mla.device_status(clear=True) == 0


def test_whole_tokens_when_cutting_is_turned_off():
    """mla_sparse_allow_cut_tokens(0): one launch per call, no buffer, same results."""
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[8192, 6000], topk=2048, seed=86)
    ref_out, ref_lse, _ = oracle.forward(inp)
    dev = to_device(inp)
    try:
        mla.allow_cut_tokens(False)
        n0 = mla.launch_count()
        out, lse, status = run_gpu(inp, dev=dev)
        assert mla.launch_count() - n0 == 1
    finally:
        mla.allow_cut_tokens(True)
    assert status == 0
    assert_out_close(out, ref_out, "whole tokens")
    assert_lse_close(lse, ref_lse, "whole tokens")
    n0 = mla.launch_count()
    out2, lse2, status2 = run_gpu(inp, dev=dev)
    assert mla.launch_count() - n0 == 2, "four tokens of 32 tiles should be cut between clusters"
    assert status2 == 0
    assert_out_close(out2, ref_out, "cut tokens")
