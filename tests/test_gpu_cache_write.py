"""GPU parity of the paged cache writer (mla_cache_write) against the oracle:
bit-exact bf16 rows, INT8 codes and fp32 scales (floating point decides the
codes, and both sides decide them with the same fp32 division and
half-to-even rounding), skipped and out-of-range indices, and the attention
kernel reading what the writer wrote."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def run_writer(inp):
    import mla_sparse_top_gb300 as mla
    dev = workloads.cache_write_to_device(inp)
    mla.mla_cache_write(dev["k_nope"], dev["k_rope"], dev["cache_index"], dev["kv_nope"], dev["kv_rope"],
                        dev["kv_scales"])
    status = mla.cache_device_status(clear=True)
    kn = dev["kv_nope"].cpu()
    kn = kn.numpy() if kn.dtype == torch.int8 else kn.view(torch.int16).numpy().view(np.uint16)
    kr = dev["kv_rope"].cpu().view(torch.int16).numpy().view(np.uint16)
    ks = dev["kv_scales"].cpu().numpy() if dev["kv_scales"] is not None else None
    return kn, kr, ks, status


def check_exact(inp):
    kn, kr, ks, status = run_writer(inp)
    on, orr, os_, bad = oracle.cache_write(inp["k_nope"], inp["k_rope"], inp["cache_index"], inp["kv_nope"],
                                           inp["kv_rope"], inp["kv_scales"])
    np.testing.assert_array_equal(kn, on)
    np.testing.assert_array_equal(kr, orr)
    if ks is not None:
        np.testing.assert_array_equal(ks.view(np.uint32), os_.view(np.uint32))
    return status, bad


@pytest.mark.parametrize("int8", [False, True])
def test_rows_scales_and_skips_bit_exact(int8):
    inp = workloads.make_cache_write_inputs(T=1000, num_blocks=16, kv_int8=int8, seed=70)
    status, bad = check_exact(inp)
    assert status == 0 and bad == 0


def test_out_of_range_index_is_skipped_and_flagged():
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_cache_write_inputs(T=40, num_blocks=2, kv_int8=True, seed=71)
    inp["cache_index"][7] = 2 * 128          # one past the last row
    inp["cache_index"][9] = 10 ** 12
    status, bad = check_exact(inp)
    assert bad == 2 and status == mla.MLA_DEVICE_BAD_BLOCK


def test_empty_write_is_a_no_op():
    inp = workloads.make_cache_write_inputs(T=0, num_blocks=1, kv_int8=True, seed=72)
    status, _ = check_exact(inp)
    assert status == 0


@pytest.mark.parametrize("maker", [workloads.cache_write_decode, workloads.cache_write_prefill])
def test_full_size_workloads_bit_exact(maker):
    status, bad = check_exact(maker())
    assert status == 0 and bad == 0


def test_attention_reads_what_the_writer_wrote():
    """Rows written by the GPU writer into an INT8 cache, then read by the
    attention kernel through the top-k lists, give the oracle's attention over
    the oracle-written cache."""
    import sys
    import os
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from gpu_util import assert_lse_close, assert_out_close, run_gpu
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[700, 1500], topk=256, seed=73, kv_int8=True)
    rows = inp["kv_nope"].shape[0]
    # new rows for positions the top-k lists use: overwrite the physical rows of some selected entries
    sel = np.unique(inp["topk_idx"][inp["topk_idx"] >= 0])[:300]
    phys = np.array([inp["block_table"][0, p // 128] * 128 + p % 128 for p in sel if p < 700], dtype=np.int64)
    w = workloads.make_cache_write_inputs(T=len(phys), num_blocks=rows // 128, kv_int8=True, seed=74, skip_every=0)
    w.update(cache_index=phys, kv_nope=inp["kv_nope"], kv_rope=inp["kv_rope"], kv_scales=inp["kv_scales"])
    kn, kr, ks, status = run_writer(w)
    assert status == 0
    on, orr, os_, _ = oracle.cache_write(w["k_nope"], w["k_rope"], phys, inp["kv_nope"], inp["kv_rope"],
                                         inp["kv_scales"])
    np.testing.assert_array_equal(kn, on)
    gpu_inp = dict(inp, kv_nope=kn, kv_rope=kr, kv_scales=ks)
    ref_inp = dict(inp, kv_nope=on, kv_rope=orr, kv_scales=os_)
    out, lse, st = run_gpu(gpu_inp)
    ref_out, ref_lse, _ = oracle.forward(ref_inp)
    assert st == 0
    assert_out_close(out, ref_out, "attention after cache write")
    assert_lse_close(lse, ref_lse, "attention after cache write")
