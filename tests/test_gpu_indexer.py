"""GPU parity of the Lightning Indexer + top-k (mla_indexer_topk) against the
oracle ("CANN DeepSeek Indexer attention", sections "Lightning Indexer" and
"Sparse Flash Attention").

Scores: fp32 on the GPU (exact bf16 products, fp32 sums over 128 dims and the
head sum) against the exact fp64 scores, within 2^-14 * M[t, j] where
M[t, j] = sum_h |w[t, h]| * sum_d |q[t, h, d] * k[j, d]| bounds every partial
sum (an fp32 sum of n terms errs by at most about n * 2^-24 of that; n <= 192).
Selection: floating point decides it, so the oracle's selection rule applied
to the GPU's own fp32 scores must give the GPU's output bit for bit; against
the exact scores every selected position must lie within the error band of
the exact k-th score, and every position clearly above it must be selected."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def bf16_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_indexer(inp):
    import mla_sparse_top_gb300 as mla
    d = inp["dims"]
    dev = workloads.indexer_to_device(inp)
    dims = mla.indexer_dims_from_workload(d)
    ws = torch.empty(mla.mla_indexer_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # NaN bytes: every position the selection reads must have been written
    dev["topk_idx"].fill_(-7)
    mla.mla_indexer_topk(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"], dev["topk_idx"], ws,
                         dims=dims)
    status = mla.indexer_device_status(clear=True)
    T, ld = d["B"] * d["S1"], d["max_blocks_per_seq"] * d["block_size"]
    scores = ws.view(torch.float32)[: T * ld].view(T, ld).cpu().numpy()
    return dev["topk_idx"].cpu().numpy(), scores, status


def magnitude(inp, tokens):
    """M[t, j] (see the module docstring) for the given tokens, all table positions."""
    d = inp["dims"]
    ld = d["max_blocks_per_seq"] * d["block_size"]
    out = np.zeros((len(tokens), ld))
    for i, t in enumerate(tokens):
        b = t // d["S1"]
        act = min(int(inp["act_seqs"][b]), ld)
        pos = np.arange(act)
        blk = inp["block_table"][b, pos // 128]
        ok = (blk >= 0) & (blk < d["num_blocks"])
        rows = np.where(ok, blk * 128 + pos % 128, 0)
        k = np.abs(bf16_f64(inp["k_cache"][rows]))               # (act, D)
        q = np.abs(bf16_f64(inp["q"][t]))                        # (H, D)
        out[i, :act] = np.abs(inp["w"][t]).astype(np.float64) @ (q @ k.T)
    return out


def check(inp, gpu_idx, gpu_sc, tokens=None, exp_status=0, status=0):
    d = inp["dims"]
    T = d["B"] * d["S1"]
    tokens = list(range(T)) if tokens is None else tokens
    ref, _ = oracle.indexer_scores(inp)
    act_of = lambda t: min(int(inp["act_seqs"][t // d["S1"]]), d["max_blocks_per_seq"] * 128)
    mag = magnitude(inp, tokens)
    tol_all = 2.0 ** -14 * mag
    for i, t in enumerate(tokens):
        n = act_of(t)
        cand = ref[t, :n] != -np.inf
        g = gpu_sc[t, :n].astype(np.float64)
        assert np.all(g[~cand] == -np.inf), f"token {t}: a non-candidate has a score"
        err = np.abs(g[cand] - ref[t, :n][cand])
        tol = tol_all[i, :n][cand] + 1e-30
        assert np.all(err <= tol), f"token {t}: score error {err.max():.3g} above {tol[err.argmax()]:.3g}"
    # the selection from the GPU's own scores, bit for bit
    sel_own = oracle.indexer_select(gpu_sc, inp["act_seqs"], d["S1"], d["topk"])
    np.testing.assert_array_equal(gpu_idx[tokens], sel_own[tokens])
    # against the exact scores: valid, and everything clearly above the threshold is in
    for i, t in enumerate(tokens):
        n = act_of(t)
        s = ref[t, :n]
        cand = np.nonzero(s != -np.inf)[0]
        k = min(d["topk"], len(cand))
        chosen = gpu_idx[t][gpu_idx[t] >= 0]
        assert len(chosen) == k and np.all(np.diff(chosen) > 0)
        assert np.all(gpu_idx[t][k:] == -1)
        if k == 0 or k == len(cand):
            np.testing.assert_array_equal(chosen, cand[:k])
            continue
        tau = np.sort(s[cand])[::-1][k - 1]
        band = 2.0 * tol_all[i, :n].max()
        assert np.all(s[chosen] >= tau - band)
        must = cand[s[cand] > tau + band]
        assert np.isin(must, chosen).all()
    assert status == exp_status


def test_tiny():
    inp = workloads.indexer_tiny()
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st)


def test_varlen():
    inp = workloads.indexer_varlen()
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st)


@pytest.mark.parametrize("S1,H", [(1, 16), (1, 64), (2, 64), (4, 64), (2, 128), (1, 256)])
def test_head_and_token_shapes(S1, H):
    inp = workloads.make_indexer_inputs(B=3, S1=S1, n_heads=H, act_seqs=[1000, 130, 2500], topk=300, seed=20 + H + S1)
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st)


def test_short_sequences_and_padding():
    inp = workloads.make_indexer_inputs(B=4, S1=2, act_seqs=[1, 127, 128, 129], topk=128, seed=30)
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st)


def test_all_scores_equal_keep_the_first_positions():
    inp = workloads.make_indexer_inputs(B=2, S1=2, act_seqs=[700, 3000], topk=256, seed=31, w_scale=0.0)
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st)
    np.testing.assert_array_equal(idx[0], np.arange(256))


def test_bad_blocks_are_skipped_and_flagged():
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_indexer_inputs(B=2, S1=2, act_seqs=[600, 600], topk=500, seed=32)
    inp["block_table"][1, 2] = 10 ** 6  # positions 256..383 of sequence 1 lose their block
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, status=st, exp_status=mla.MLA_DEVICE_BAD_BLOCK)
    assert not np.isin(np.arange(256, 384), idx[2]).any()


def test_permuted_blocks_give_identical_output():
    inp = workloads.make_indexer_inputs(B=2, S1=2, act_seqs=[900, 1200], topk=200, seed=33, poison_unused=False)
    idx, sc, _ = run_indexer(inp)
    nb = inp["dims"]["num_blocks"]
    perm = np.random.default_rng(1).permutation(nb)
    cache2 = np.empty_like(inp["k_cache"])
    for old in range(nb):
        cache2[perm[old] * 128:(perm[old] + 1) * 128] = inp["k_cache"][old * 128:(old + 1) * 128]
    inp2 = dict(inp, k_cache=cache2,
                block_table=np.where(inp["block_table"] >= 0, perm[inp["block_table"]], -1).astype(np.int32))
    idx2, sc2, _ = run_indexer(inp2)
    np.testing.assert_array_equal(idx, idx2)
    np.testing.assert_array_equal(sc[:, :900], sc2[:, :900])


def test_full_size_decode_sampled_tokens():
    inp = workloads.indexer_decode()
    idx, sc, st = run_indexer(inp)
    check(inp, idx, sc, tokens=[0, 1, 63, 64, 126, 127], status=st)


def test_split_phases_equal_the_combined_call():
    import mla_sparse_top_gb300 as mla
    inp = workloads.make_indexer_inputs(B=3, S1=2, act_seqs=[5000, 300, 2049], topk=1024, seed=34)
    idx, sc, _ = run_indexer(inp)
    d = inp["dims"]
    dev = workloads.indexer_to_device(inp)
    dims = mla.indexer_dims_from_workload(d)
    scores = torch.empty(mla.mla_indexer_workspace_bytes(dims) // 4, dtype=torch.float32, device="cuda")
    mla.mla_indexer_scores(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"], scores, dims=dims)
    mla.mla_indexer_select(scores, dev["act_seqs"], dev["topk_idx"], dims=dims)
    assert mla.indexer_device_status(clear=True) == 0
    np.testing.assert_array_equal(dev["topk_idx"].cpu().numpy(), idx)
    T, ld = d["B"] * d["S1"], d["max_blocks_per_seq"] * 128
    for t in range(T):
        n = int(inp["act_seqs"][t // 2])
        np.testing.assert_array_equal(scores.view(T, ld)[t, :n].cpu().numpy(), sc[t, :n])


@pytest.mark.parametrize("kind", ["coarse_ties", "signed_zeros", "sparse_candidates", "all_equal", "extremes"])
def test_selection_phase_on_given_scores(kind):
    """The selection kernel alone on fp32 scores built here, against the
    oracle's selection rule on the same fp32 values."""
    import mla_sparse_top_gb300 as mla
    rng = np.random.default_rng(40)
    B, S1, W, topk = 4, 2, 40, 700
    ld = W * 128
    act = np.array([ld, 5000, 699, 1], dtype=np.int32)
    T = B * S1
    if kind == "coarse_ties":
        sc = rng.integers(-20, 20, size=(T, ld)).astype(np.float32)            # many exact ties
    elif kind == "signed_zeros":
        sc = np.where(rng.random((T, ld)) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        sc[:, ::7] = 1.0
    elif kind == "sparse_candidates":
        sc = rng.standard_normal((T, ld)).astype(np.float32)
        sc[rng.random((T, ld)) < 0.9] = -np.inf                                 # ~10% candidates
    elif kind == "all_equal":
        sc = np.full((T, ld), 3.5, dtype=np.float32)
    else:
        sc = rng.choice(np.array([np.finfo(np.float32).max, -np.finfo(np.float32).max, np.finfo(np.float32).tiny,
                                  -np.finfo(np.float32).tiny, 1e-45, -1e-45, 0.0, 1.0], dtype=np.float32),
                        size=(T, ld))
    sc = np.ascontiguousarray(sc, dtype=np.float32)
    d = dict(B=B, S1=S1, n_heads=64, head_dim=128, block_size=128, num_blocks=W, max_blocks_per_seq=W, topk=topk)
    dims = mla.indexer_dims_from_workload(d)
    dev_sc = torch.from_numpy(sc).cuda()
    dev_act = torch.from_numpy(act).cuda()
    out = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    mla.mla_indexer_select(dev_sc, dev_act, out, dims=dims)
    assert mla.indexer_device_status(clear=True) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.indexer_select(sc, act, S1, topk))


@pytest.mark.parametrize("kind", ["gaussian", "coarse_ties"])
def test_selection_phase_on_rows_longer_than_one_round(kind):
    """Rows of more than 8192 positions: the later positions are re-read from
    the scores on every pass."""
    import mla_sparse_top_gb300 as mla
    rng = np.random.default_rng(41)
    B, S1, W, topk = 4, 1, 160, 2048
    ld = W * 128
    act = np.array([ld, 9000, 8193, 8192], dtype=np.int32)
    sc = rng.standard_normal((B, ld)).astype(np.float32)
    if kind == "coarse_ties":
        sc = np.round(sc * 4).astype(np.float32)
    d = dict(B=B, S1=S1, n_heads=64, head_dim=128, block_size=128, num_blocks=W, max_blocks_per_seq=W, topk=topk)
    dims = mla.indexer_dims_from_workload(d)
    out = torch.full((B, topk), -7, dtype=torch.int32, device="cuda")
    mla.mla_indexer_select(torch.from_numpy(sc).cuda(), torch.from_numpy(act).cuda(), out, dims=dims)
    assert mla.indexer_device_status(clear=True) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.indexer_select(sc, act, S1, topk))
