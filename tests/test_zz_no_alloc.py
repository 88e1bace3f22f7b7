"""mla_indexer_topk_noalloc against mla_indexer_topk: two calls in a row with
different inputs, each compared with the workspace entry point on the same
inputs (a stale or shared scratch would show in the second call)."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _call_both(inp):
    import mla_sparse_top_gb300 as mla
    d = inp["dims"]
    dev = workloads.indexer_to_device(inp)
    dims = mla.indexer_dims_from_workload(d)
    ws = torch.empty(mla.mla_indexer_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    ref = torch.full_like(dev["topk_idx"], -7)
    mla.mla_indexer_topk(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"], ref, ws, dims=dims)
    out = torch.full_like(dev["topk_idx"], -7)
    mla.mla_indexer_topk_noalloc(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"], out,
                                 dims=dims)
    assert mla.indexer_device_status(clear=True) == 0
    return ref.cpu().numpy(), out.cpu().numpy()


def test_noalloc_equals_the_workspace_entry_point_on_two_calls_in_a_row():
    first = workloads.make_indexer_inputs(B=8, S1=2, act_seqs=[8192, 300, 5000, 129, 8192, 7000, 4096, 2049],
                                          topk=2048, seed=60)
    second = workloads.make_indexer_inputs(B=6, S1=1, act_seqs=[1000, 8192, 64, 3000, 128, 6000], topk=512,
                                           seed=61)
    for inp in (first, second):
        ref, out = _call_both(inp)
        np.testing.assert_array_equal(out, ref)
        assert (out[:, 0] >= 0).all()


def test_noalloc_largest_accepted_size():
    """B * S1 * W * 128 = 2 Mi scores, the stated limit."""
    inp = workloads.make_indexer_inputs(B=16, S1=2, act_seqs=[8192] * 16, topk=2048, seed=62, n_heads=64,
                                        max_blocks_per_seq=512)
    assert inp["dims"]["B"] * inp["dims"]["S1"] * inp["dims"]["max_blocks_per_seq"] * 128 == 2 << 20
    ref, out = _call_both(inp)
    np.testing.assert_array_equal(out, ref)
