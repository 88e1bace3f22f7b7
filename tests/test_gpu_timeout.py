"""The bounded device waits of the attention kernel.

Every wait of the kernel gives up after a bound (mla_sparse_set_wait_limit_ns,
500 ms by default) instead of spinning forever; the launch then leaves its
roles, drains its copies and MMAs, frees its tensor memory and raises
MLA_DEVICE_TIMEOUT in the device status word.  Here the bound is cut to 1 us,
far below the first gather's latency, so a wait runs out on purpose (nothing
on the GPU is made to fail: the work is only slower than the bound).  The
status must show the timeout; after clearing it and restoring the bound, the
next call on the same inputs must match the oracle.
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
