"""A decode step through two of the library's calls, as a user chains them:
mla_prolog turns hidden states into the absorbed query and writes each
token's key row into the paged cache at its own position, then
mla_sparse_attn_fwd attends over that cache with top-k lists that include
the new positions.  The oracle runs the same chain on its own (prolog oracle
-> its cache and its query rounded to bf16 -> attention oracle).

Tolerance: the two chains differ only where the prolog's bf16 roundings do
(the prolog tests bound that at 2.5e-3 of the query's RMS overall, and the
cache rows at one bf16 unit or half an INT8 step).  The prolog's normalised
keys are long (|k| ~ 24), so at softmax_scale 1/sqrt(576) a token's few new
rows carry nearly all the weight and any difference in q is amplified; the
chain runs at 0.05/sqrt(576), where even noise of 2.5e-3 rms on every q
element (far more than the rare rounding flips) stays below 0.4 of the bound
|gpu - oracle| <= 1e-2 |oracle| + 1e-2 rms(row) in the oracle itself.  A
layout or indexing mistake moves the output by O(rms).  Each call's own
parity, at the operator's tolerance, is in its own test file."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import prolog as P

pytestmark = pytest.mark.gpu


def chain_inputs(kv_int8, seed):
    B, S1, H = 2, 2, 128
    act = np.array([300, 700], dtype=np.int32)
    inp = workloads.make_prolog_inputs(T=B * S1, seed=seed, hidden=256, q_lora=128, n_heads=H, num_blocks=16,
                                       kv_int8=kv_int8)
    rng = np.random.default_rng(seed)
    W = 8
    bt = np.full((B, W), -1, dtype=np.int32)
    phys = rng.permutation(16).astype(np.int32)
    bt[0, :3], bt[1, :6] = phys[:3], phys[3:9]
    topk = 160
    lists = np.empty((B * S1, topk), dtype=np.int32)
    idx = np.empty(B * S1, dtype=np.int64)
    for t in range(B * S1):
        b, s = divmod(t, S1)
        p = int(act[b]) - S1 + s                       # the token's own position
        idx[t] = int(bt[b, p // 128]) * 128 + p % 128
        others = rng.choice(np.setdiff1d(np.arange(act[b]), [p]), topk - 1, replace=False)
        lists[t] = rng.permutation(np.concatenate([[p], others]))
    inp["cache_index"] = idx
    return inp, dict(B=B, S1=S1, H=H, act=act, bt=bt, lists=lists, topk=topk)


@pytest.mark.parametrize("kv_int8", [False, True])
def test_prolog_then_attention_matches_the_oracle_chain(kv_int8):
    import mla_sparse_top_gb300 as mla
    inp, c = chain_inputs(kv_int8, seed=60 + int(kv_int8))
    scale = 0.05 * 576 ** -0.5
    # ---- GPU chain
    dev = workloads.prolog_to_device(inp)
    T, H = c["B"] * c["S1"], c["H"]
    q_nope = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    q_rope = torch.empty((T, H, 64), dtype=torch.bfloat16, device="cuda")
    dims = mla.prolog_dims(dev["x"], dev["wq_a"], dev["wq_b"], dev["kv_nope"])
    ws = torch.empty(mla.mla_prolog_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    mla.mla_prolog(dev["x"], dev["wq_a"], dev["gamma_cq"], dev["wq_b"], dev["w_uk"], dev["wkv"], dev["gamma_ckv"],
                   dev["cos"], dev["sin"], dev["cache_index"], q_nope, q_rope, dev["kv_nope"], dev["kv_rope"],
                   dev["kv_scales"], ws, dims=dims)
    assert mla.prolog_device_status(clear=True) == 0
    out = torch.empty_like(q_nope)
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    mla.mla_sparse_attn_fwd(q_nope, q_rope, dev["kv_nope"], dev["kv_rope"], dev["kv_scales"], t32(c["lists"]),
                            t32(c["bt"]), t32(c["act"]), out, lse, softmax_scale=scale, S1=c["S1"])
    assert mla.device_status(clear=True) == 0
    g_out = out.float().cpu().numpy().astype(np.float64)
    g_lse = lse.cpu().numpy().astype(np.float64)
    # ---- oracle chain
    ref, (kn, kr, ks, bad) = P.forward_with_cache(inp)
    assert bad == 0
    att = dict(q_nope=P.f64_to_bf16_bits(ref["q_nope"]), q_rope=P.f64_to_bf16_bits(ref["q_rope"]), kv_nope=kn,
               kv_rope=kr, kv_scales=ks, topk_idx=c["lists"], block_table=c["bt"], act_seqs=c["act"],
               softmax_scale=scale,
               dims=dict(B=c["B"], S1=c["S1"], n_q=H, n_kv=1, d_nope=512, d_rope=64, block_size=128,
                         num_blocks=16, max_blocks_per_seq=c["bt"].shape[1], topk=c["topk"], kv_int8=int(kv_int8)))
    r_out, r_lse, r_bad = oracle.forward(att)
    assert r_bad == 0
    rms = np.sqrt(np.mean(r_out ** 2, axis=-1, keepdims=True))
    err = np.abs(g_out - r_out)
    assert np.all(err <= 1e-2 * np.abs(r_out) + 1e-2 * rms), float(np.max(err / (np.abs(r_out) + rms)))
    np.testing.assert_allclose(g_lse, r_lse, rtol=1e-2, atol=1e-2)
