"""GPU parity of sliding-window attention (mla_swa_fwd) with the oracle
(window lists + the attention definition), at the stated tolerance."""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import assert_lse_close, assert_out_close, bf16_to_f64, dims_of, to_device  # noqa: E402


def run_swa(inp, window):
    import mla_sparse_top_gb300 as mla
    dev = to_device(inp)
    dev["out"].fill_(float("nan"))
    dev["lse"].fill_(float("nan"))
    d = dims_of(inp)
    d.topk = 0  # ignored by the window entry point
    mla.mla_swa_fwd(dev["q_nope"], dev["q_rope"], dev["kv_nope"], dev["kv_rope"], dev["kv_scales"],
                    dev["block_table"], dev["act_seqs"], dev["out"], dev["lse"], window=window,
                    softmax_scale=inp["softmax_scale"], mode=inp.get("mode", "decode"), dims=d)
    status = mla.device_status(clear=True)
    out = bf16_to_f64(dev["out"].view(torch.int16).cpu().numpy().view(np.uint16))
    return out, dev["lse"].cpu().numpy().astype(np.float64), status


@pytest.mark.parametrize("window,S1,kv_int8", [(1, 1, False), (7, 2, False), (64, 2, True), (100, 2, False),
                                                (130, 3, True), (1000, 2, False)])
def test_window_attention(window, S1, kv_int8):
    inp = workloads.make_inputs(B=5, S1=S1, n_q=128, act_seqs=[1, 40, 300, 1500, 129], topk=16, seed=100 + window,
                                kv_int8=kv_int8)
    out, lse, status = run_swa(inp, window)
    ref_out, ref_lse, _ = oracle.swa_forward(inp, window)
    assert status == 0
    assert_out_close(out, ref_out, f"swa w={window}")
    assert_lse_close(lse, ref_lse, f"swa w={window}")


@pytest.mark.parametrize("window", [128, 2048])
def test_decode_full_size_sampled(window):
    inp = workloads.make_inputs(B=64, S1=2, n_q=128, act_seqs=[8192] * 64, topk=16, seed=110)
    out, lse, status = run_swa(inp, window)
    toks = [0, 1, 63, 64, 126, 127]
    ref_out, ref_lse, _ = oracle.swa_forward(inp, window, tokens=toks)
    assert status == 0 and np.isfinite(out).all()
    assert_out_close(out[toks], ref_out, f"swa decode w={window}")
    assert_lse_close(lse[toks], ref_lse, f"swa decode w={window}")


def test_prefill_window():
    inp = workloads.make_inputs(B=2, S1=256, n_q=64, act_seqs=[2048, 700], topk=16, seed=111, mode="prefill")
    out, lse, status = run_swa(inp, 512)
    ref_out, ref_lse, _ = oracle.swa_forward(inp, 512)
    assert status == 0
    assert_out_close(out, ref_out, "swa prefill")
    assert_lse_close(lse, ref_lse, "swa prefill")
