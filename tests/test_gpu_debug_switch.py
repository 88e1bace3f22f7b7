"""The MLA_SPARSE_DEBUG switch of the binding: with it set, a call whose
kernel raised a device status bit (here a bad block id in the attention's
block table, and a cache index past the cache) fails at once with
MLA_ERR_DEVICE_STATUS, and the status word is cleared; clean calls pass."""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu


def test_attention_bad_block_raises_under_the_switch(monkeypatch):
    import mla_sparse_top_gb300 as mla
    from gpu_util import launch, to_device
    inp = workloads.make_inputs(B=2, S1=2, n_q=128, act_seqs=[600, 300], topk=150, seed=30)
    dev = to_device(inp)
    mla.device_status(clear=True)  # no bit left over from an earlier test
    monkeypatch.setenv("MLA_SPARSE_DEBUG", "1")
    launch(inp, dev)  # a clean call passes
    inp["block_table"][0, 1] = 10 ** 6
    dev = to_device(inp)
    with pytest.raises(mla.MlaError) as e:
        launch(inp, dev)
    assert e.value.status == -7 and "MLA_SPARSE_DEBUG" in str(e.value)
    assert mla.device_status(clear=True) == 0  # the switch cleared the word


def test_cache_write_bad_index_raises_under_the_switch(monkeypatch):
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_cache_write_inputs(T=40, num_blocks=2, kv_int8=True, seed=71)
    dev = workloads.cache_write_to_device(inp)
    mla.cache_device_status(clear=True)  # no bit left over from an earlier test
    monkeypatch.setenv("MLA_SPARSE_DEBUG", "1")
    mla.mla_cache_write(dev["k_nope"], dev["k_rope"], dev["cache_index"], dev["kv_nope"], dev["kv_rope"],
                        dev["kv_scales"])
    bad = inp["cache_index"].copy()
    bad[7] = 2 * 128
    import torch
    dev["cache_index"] = torch.from_numpy(np.ascontiguousarray(bad)).cuda()
    with pytest.raises(mla.MlaError) as e:
        mla.mla_cache_write(dev["k_nope"], dev["k_rope"], dev["cache_index"], dev["kv_nope"], dev["kv_rope"],
                            dev["kv_scales"])
    assert e.value.status == -7
    monkeypatch.delenv("MLA_SPARSE_DEBUG")
    assert mla.cache_device_status(clear=True) == 0
