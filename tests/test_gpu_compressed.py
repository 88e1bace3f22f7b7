"""GPU parity of compressed / sparse compressed flash attention
(mla_compressed_attn_fwd) with the numpy oracle (oracle.compressed), at the
stated tolerance."""
import numpy as np
import pytest

import oracle.compressed as comp
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gpu_util import assert_lse_close, assert_out_close, bf16_to_f64, dims_of, to_device  # noqa: E402


def run_compressed(inp):
    import mla_sparse_top_gb300 as mla
    d = inp["dims"]
    dev = to_device(inp)
    dev["out"].fill_(float("nan"))
    dev["lse"].fill_(float("nan"))

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    def raw(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()

    cmp_nope = raw(inp["cmp_nope"]) if d["kv_int8"] else bf(inp["cmp_nope"])
    mla.mla_compressed_attn_fwd(dev["q_nope"], dev["q_rope"], dev["kv_nope"], dev["kv_rope"], dev["kv_scales"],
                                dev["block_table"], cmp_nope, bf(inp["cmp_rope"]), raw(inp.get("cmp_scales")),
                                raw(inp["cmp_block_table"]), dev["act_seqs"], dev["out"], dev["lse"],
                                window=d["window"], cmp_ratio=d["cmp_ratio"], cmp_idx=raw(inp.get("cmp_idx")),
                                softmax_scale=inp["softmax_scale"], mode=inp.get("mode", "decode"),
                                dims=dims_of(inp))
    status = mla.device_status(clear=True)
    out = bf16_to_f64(dev["out"].view(torch.int16).cpu().numpy().view(np.uint16))
    return out, dev["lse"].cpu().numpy().astype(np.float64), status


def check(inp, label, tokens=None):
    d = inp["dims"]
    out, lse, status = run_compressed(inp)
    ref_out, ref_lse, bad = comp.forward(inp, d["window"], d["cmp_ratio"], cmp_idx=inp.get("cmp_idx"), tokens=tokens)
    if tokens is not None:
        out, lse = out[tokens], lse[tokens]
    else:
        assert status == (1 if bad else 0), f"{label}: status {status:#x}, oracle bad {bad}"
    assert_out_close(out, ref_out, label)
    assert_lse_close(lse, ref_lse, label)
    return status


@pytest.mark.parametrize("ratio,topk,kv_int8", [(4, None, False), (4, 40, False), (128, None, True), (1, 100, True),
                                                 (8, 7, False)])
def test_cfa_and_scfa(ratio, topk, kv_int8):
    inp = workloads.make_compressed_inputs(B=4, S1=2, n_q=128, act_seqs=[1, 300, 1100, 129], window=48,
                                           cmp_ratio=ratio, cmp_topk=topk, seed=130 + ratio, kv_int8=kv_int8)
    check(inp, f"ratio={ratio} topk={topk} int8={kv_int8}")


def test_bad_compressed_block_is_masked_and_flagged():
    inp = workloads.make_compressed_inputs(B=2, S1=2, n_q=64, act_seqs=[700, 900], window=32, cmp_ratio=2,
                                           cmp_topk=None, seed=140)
    inp["cmp_block_table"][1, 1] = 10 ** 6                 # entries 128..255 of sequence 1 lose their block
    status = check(inp, "bad compressed block")
    assert status == 1


@pytest.mark.parametrize("name", ["cfa_decode", "scfa_decode"])
def test_full_size_sampled(name):
    inp = workloads.COMPRESSED_NAMED[name]()
    check(inp, name, tokens=[0, 1, 63, 64, 126, 127])
