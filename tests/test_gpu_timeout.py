"""The bounded device waits of the attention kernel.

Every wait of the kernel gives up after a bound (mla_sparse_set_wait_limit_ns,
500 ms by default) instead of spinning forever; the launch then leaves its
roles, drains its copies and MMAs, frees its tensor memory and raises
MLA_DEVICE_TIMEOUT in the device status word.  Here the bound is cut to 1 us,
far below the first gather's latency, so a wait runs out on purpose (nothing
on the GPU is made to fail: the work is only slower than the bound).  The
status must show the timeout; after clearing it and restoring the bound, the
next call on the same inputs must match the oracle.  The Lightning Indexer's
score kernel and the MLA Prolog's product kernel take the same bound: for them
the call after the timeout must repeat, bit for bit, a call made before it.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import assert_lse_close, assert_out_close, launch, run_gpu, to_device  # noqa: E402


# B=64 S1=2 runs whole tokens per cluster; B=15 S1=2 (30 tokens of 32 tiles)
# cuts tokens between clusters, so a launch that gives up leaves arrival
# counts behind that the next launch must ignore.
@pytest.mark.parametrize("name, B, topk, kv_int8", [("mtp", 64, 512, False), ("mtp", 64, 512, True),
                                                    ("mtp", 15, 2048, False), ("swa", 64, 512, False)])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_exact(name, B, topk, kv_int8):
    import mla_sparse_top_gb300 as mla
    acts = [4000, 2500, 700, 8000]
    inp = workloads.make_inputs(B=B, S1=2, n_q=128, act_seqs=[acts[b % 4] for b in range(B)], topk=topk, seed=70,
                                kv_int8=kv_int8)
    dev = to_device(inp)
    assert mla.device_status(clear=True) == 0
    mla.set_wait_limit_ns(1000)
    try:
        if name == "swa":
            mla.mla_swa_fwd(dev["q_nope"], dev["q_rope"], dev["kv_nope"], dev["kv_rope"], dev["kv_scales"],
                            dev["block_table"], dev["act_seqs"], dev["out"], dev["lse"], window=300,
                            softmax_scale=inp["softmax_scale"], dims=mla.dims_from_workload(inp["dims"]))
        else:
            launch(inp, dev)
        status = mla.device_status(clear=True)
    finally:
        mla.set_wait_limit_ns(mla.DEFAULT_WAIT_LIMIT_NS)
    assert status & mla.MLA_DEVICE_TIMEOUT, f"status {status:#x}: no wait ran out under a 1 us bound"
    # the context is intact and the next launch does the whole job again
    out, lse, status = run_gpu(inp, dev=dev)
    assert status == 0, f"status {status:#x} after the bound was restored"
    ref_out, ref_lse, _ = oracle.forward(inp)
    assert_out_close(out, ref_out, f"{name} B={B} int8={kv_int8} after a timeout")
    assert_lse_close(lse, ref_lse, f"{name} B={B} int8={kv_int8} after a timeout")
    assert np.isfinite(out).all()


def _flush_l2():
    # a write larger than L2, so that the next call's first loads come from HBM
    torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda").fill_(1.0)
    torch.cuda.synchronize()


def test_indexer_wait_that_runs_out_is_reported_and_the_next_call_is_identical():
    """The Lightning Indexer's score kernel takes the same bound: a 1 us bound
    makes its waits run out, the status shows it, and after restoring the
    bound the next call gives the same selection bit for bit."""
    import mla_sparse_top_gb300 as mla
    inp = workloads.INDEXER_NAMED["indexer_decode"]()
    dev = workloads.indexer_to_device(inp)
    dims = mla.indexer_dims_from_workload(inp["dims"])
    ws = torch.empty(mla.mla_indexer_workspace_bytes(dims), dtype=torch.uint8, device="cuda")

    def call():
        dev["topk_idx"].fill_(-7)
        mla.mla_indexer_topk(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"],
                             dev["topk_idx"], ws, dims=dims)
        return mla.indexer_device_status(clear=True), dev["topk_idx"].cpu().numpy().copy()

    status, ref = call()
    assert status == 0
    _flush_l2()
    mla.set_wait_limit_ns(1000)
    try:
        status, _ = call()
    finally:
        mla.set_wait_limit_ns(mla.DEFAULT_WAIT_LIMIT_NS)
    assert status & mla.MLA_DEVICE_TIMEOUT, f"status {status:#x}: no wait ran out under a 1 us bound"
    status, again = call()
    assert status == 0
    np.testing.assert_array_equal(again, ref)


def test_prolog_wait_that_runs_out_is_reported_and_the_next_call_is_identical():
    """The MLA Prolog's product kernel takes the same bound (decode size: its
    weights, 123 MB, stream from HBM)."""
    import mla_sparse_top_gb300 as mla
    inp = workloads.PROLOG_NAMED["prolog_decode"]()
    dev = workloads.prolog_to_device(inp)
    d = inp["dims"]
    T, H = d["T"], d["n_heads"]
    q_nope = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    q_rope = torch.empty((T, H, 64), dtype=torch.bfloat16, device="cuda")
    dims = mla.prolog_dims(dev["x"], dev["wq_a"], dev["wq_b"], dev["kv_nope"])
    ws = torch.empty(mla.mla_prolog_workspace_bytes(dims), dtype=torch.uint8, device="cuda")

    def call():
        q_nope.fill_(float("nan"))
        mla.mla_prolog(dev["x"], dev["wq_a"], dev["gamma_cq"], dev["wq_b"], dev["w_uk"], dev["wkv"], dev["gamma_ckv"],
                       dev["cos"], dev["sin"], dev["cache_index"], q_nope, q_rope, dev["kv_nope"], dev["kv_rope"],
                       dev["kv_scales"], ws, dims=dims)
        return (mla.prolog_device_status(clear=True), q_nope.view(torch.int16).cpu().numpy().copy(),
                q_rope.view(torch.int16).cpu().numpy().copy())

    status, ref_n, ref_r = call()
    assert status == 0
    _flush_l2()
    mla.set_wait_limit_ns(1000)
    try:
        status, _, _ = call()
    finally:
        mla.set_wait_limit_ns(mla.DEFAULT_WAIT_LIMIT_NS)
    assert status & mla.MLA_DEVICE_TIMEOUT, f"status {status:#x}: no wait ran out under a 1 us bound"
    status, n2, r2 = call()
    assert status == 0
    np.testing.assert_array_equal(n2, ref_n)
    np.testing.assert_array_equal(r2, ref_r)
