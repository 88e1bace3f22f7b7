"""GPU parity of the MLA Prolog (mla_prolog) against the oracle.

Tolerances, from the arithmetic: the GPU accumulates the products in fp32
and rounds c^Q, the pre-absorption query and the outputs to bf16 (8
significant bits), as the oracle does at the same storage points in fp64.
fp32 accumulation moves a stored value by ~1e-6 of its row's scale, so about
one c^Q element in a thousand (~1.5 per token) rounds the other way (one
unit, 2^-8..2^-7 relative).  Each such flip shifts the token's q = c^Q @ wq_b
by ~2e-4 of its RMS, which makes a few of each head's 128 pre-absorption
values round the other way too; through the 128-long absorption each moves
an output by up to ~2^-7 * |q_i| * |w_uk| (~1e-3 of the row's RMS, a few
times that in the tails).  Hence, for q_nope,
    per element   |gpu - oracle| <= 2^-7 |oracle| + 2e-2 rms(row)
    overall       rms(gpu - oracle) <= 2.5e-3 rms(oracle)
(a wrong index, sign or term moves elements by O(rms), far outside both);
q_rope has no stored intermediate of its own: 2^-7 |oracle| + 6e-3 rms(row).
The oracle's outputs are exact, the GPU's rounded once (bf16 rounding alone
gives an overall relative RMS error near 8e-4).  Cache rows: the bf16 key row
is within 2^-8 |k| + 1e-4 rms(row) of the exact key and equals the oracle's
rounded bits almost everywhere; INT8 codes dequantise to within half a step
(scale / 2) plus the bf16 rounding, and equal the oracle's codes almost
everywhere.  Rows not written stay bit for bit."""
import numpy as np
import pytest
import torch

import workloads
from oracle import prolog as P

pytestmark = pytest.mark.gpu


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_prolog(inp, dev=None):
    import mla_sparse_top_gb300 as mla
    dev = dev or workloads.prolog_to_device(inp)
    d = inp["dims"]
    T, H = d["T"], d["n_heads"]
    q_nope = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    q_rope = torch.empty((T, H, 64), dtype=torch.bfloat16, device="cuda")
    dims = mla.prolog_dims(dev["x"], dev["wq_a"], dev["wq_b"], dev["kv_nope"])
    ws = torch.empty(mla.mla_prolog_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    mla.mla_prolog(dev["x"], dev["wq_a"], dev["gamma_cq"], dev["wq_b"], dev["w_uk"], dev["wkv"], dev["gamma_ckv"],
                   dev["cos"], dev["sin"], dev["cache_index"], q_nope, q_rope, dev["kv_nope"], dev["kv_rope"],
                   dev["kv_scales"], ws, dims=dims)
    status = mla.prolog_device_status(clear=True)
    return dict(q_nope=q_nope, q_rope=q_rope, dev=dev, ws=ws, dims=dims, status=status)


def rms(a):
    return np.sqrt(np.mean(a * a, axis=-1, keepdims=True))


def assert_close_rows(gpu, ref, what, rel=2.0 ** -7, row_frac=6e-3):
    err = np.abs(gpu - ref)
    bound = rel * np.abs(ref) + row_frac * rms(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance, worst excess "
                           f"{float(np.max(err - bound)):.3g}")


def assert_overall(gpu, ref, what, frac=2.5e-3):
    e = float(np.sqrt(np.mean((gpu - ref) ** 2)))
    r = float(np.sqrt(np.mean(ref ** 2)))
    assert e <= frac * r, f"{what}: overall relative RMS error {e / max(r, 1e-300):.3g} > {frac}"


def check(inp, res):
    ref, (kn_ref, kr_ref, ks_ref, bad_ref) = P.forward_with_cache(inp)
    qn, qr = bf16_to_f64(res["q_nope"]), bf16_to_f64(res["q_rope"])
    assert_close_rows(qn, ref["q_nope"], "q_nope", row_frac=2e-2)
    assert_overall(qn, ref["q_nope"], "q_nope")
    assert_close_rows(qr, ref["q_rope"], "q_rope")
    assert_overall(qr, ref["q_rope"], "q_rope")
    dev = res["dev"]
    int8 = inp["dims"]["kv_int8"]
    kr = dev["kv_rope"].cpu().view(torch.int16).numpy().view(np.uint16)
    if int8:
        kn = dev["kv_nope"].cpu().numpy()
        ks = dev["kv_scales"].cpu().numpy()
    else:
        kn = dev["kv_nope"].cpu().view(torch.int16).numpy().view(np.uint16)
        ks = None
    idx = inp["cache_index"]
    rows = idx[(idx >= 0) & (idx < kn.shape[0])]
    untouched = np.setdiff1d(np.arange(kn.shape[0]), rows)
    np.testing.assert_array_equal(kn[untouched], inp["kv_nope"][untouched])
    np.testing.assert_array_equal(kr[untouched], inp["kv_rope"][untouched])
    toks = np.nonzero((idx >= 0) & (idx < kn.shape[0]))[0]
    if len(toks) == 0:
        return ref
    r = idx[toks]
    k_exact = ref["k_nope_exact"][toks]
    kr_exact = ref["k_rope_exact"][toks]
    assert_close_rows(P.bf16_to_f64(kr[r]), kr_exact, "k_rope", rel=2.0 ** -8, row_frac=1e-4)
    assert np.mean(kr[r] == kr_ref[r]) >= 0.99
    if not int8:
        assert_close_rows(P.bf16_to_f64(kn[r]), k_exact, "k_nope", rel=2.0 ** -8, row_frac=1e-4)
        assert np.mean(kn[r] == kn_ref[r]) >= 0.99
    else:
        sc = np.repeat(ks[r].astype(np.float64), 128, axis=1)
        dq = kn[r].astype(np.float64) * sc
        bound = 0.5 * sc * (1 + 1e-6) + 2.0 ** -8 * np.abs(k_exact) + 1e-4 * rms(k_exact)
        assert np.all(np.abs(dq - k_exact) <= bound), "INT8 codes out of half a step of the exact key"
        assert np.mean(kn[r] == kn_ref[r]) >= 0.99
        np.testing.assert_allclose(ks[r], ks_ref[r], rtol=2.0 ** -7)
    return ref


def test_tiny_bf16_cache_with_skipped_rows_zero_row_and_scaled_row():
    inp = workloads.prolog_tiny()
    res = run_prolog(inp)
    assert res["status"] == 0
    check(inp, res)
    assert torch.count_nonzero(res["q_nope"][1]) == 0          # the zero hidden row stays exactly zero


def test_decode_128_tokens_int8_cache():
    inp = workloads.prolog_decode()
    res = run_prolog(inp)
    assert res["status"] == 0
    check(inp, res)


def test_prefill_1000_tokens_bf16_cache():
    inp = workloads.prolog_prefill()
    res = run_prolog(inp)
    assert res["status"] == 0
    check(inp, res)


@pytest.mark.parametrize("T,H,hidden,q_lora,int8", [(1, 1, 64, 32, True), (3, 5, 136, 40, False),
                                                    (33, 16, 7168, 1536, True)])
def test_odd_shapes(T, H, hidden, q_lora, int8):
    inp = workloads.make_prolog_inputs(T=T, seed=20 + T, hidden=hidden, q_lora=q_lora, n_heads=H, num_blocks=2,
                                       kv_int8=int8)
    res = run_prolog(inp)
    assert res["status"] == 0
    check(inp, res)


def test_out_of_range_cache_index_is_skipped_and_flagged():
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_prolog_inputs(T=6, seed=30, hidden=64, q_lora=32, n_heads=2, num_blocks=1, kv_int8=True)
    inp["cache_index"][2] = 128                                # one past the last row
    res = run_prolog(inp)
    assert res["status"] == mla.MLA_DEVICE_BAD_BLOCK
    check(inp, res)


def test_empty_call_is_a_no_op():
    inp = workloads.make_prolog_inputs(T=0, seed=31, hidden=64, q_lora=32, n_heads=2, num_blocks=1)
    res = run_prolog(inp)
    assert res["status"] == 0


def test_graph_capture_replays_the_same_outputs():
    import mla_sparse_top_gb300 as mla
    inp = workloads.prolog_tiny(seed=32)
    res = run_prolog(inp)                                      # the first call sets up the stream, events and handle
    dev, dims, ws = res["dev"], res["dims"], res["ws"]
    q1, r1 = res["q_nope"].clone(), res["q_rope"].clone()
    kv1 = dev["kv_nope"].clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mla.mla_prolog(dev["x"], dev["wq_a"], dev["gamma_cq"], dev["wq_b"], dev["w_uk"], dev["wkv"],
                       dev["gamma_ckv"], dev["cos"], dev["sin"], dev["cache_index"], res["q_nope"], res["q_rope"],
                       dev["kv_nope"], dev["kv_rope"], dev["kv_scales"], ws, dims=dims)
    res["q_nope"].zero_()
    res["q_rope"].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(res["q_nope"], q1) and torch.equal(res["q_rope"], r1)
    assert torch.equal(dev["kv_nope"], kv1)
