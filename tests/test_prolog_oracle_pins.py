"""Pins of the MLA Prolog oracle ("NPU DeepSeek-V4 PyPTO fused-operator
optimization", section MlaProlog; "CANN DeepSeek Indexer attention", section
MLA Prolog): bf16 rounding against torch's conversion and hand-worked ties,
RMSNorm and RoPE closed forms (RoPE as complex multiplication), the
relative-position property of RoPE, a whole-prolog closed form with
selection-matrix weights, head permutation, absorption as associativity, and
the cache write.  CPU only."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import cache_write
from oracle import prolog as P


def bf16_bits_of(v):
    return workloads._bf16_bits(torch.tensor(np.asarray(v, dtype=np.float32)))


# ------------------------------------------------------------------ bf16 rounding
def test_round_bf16_hand_worked_ties():
    # bf16 keeps 8 significant bits: the spacing just above 1 is 2^-7
    assert P.round_bf16(1.0 + 2.0 ** -8) == 1.0                    # tie -> even (1)
    assert P.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6    # tie -> even (mantissa 2)
    assert P.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7   # just above a tie rounds up
    assert P.round_bf16(-(1.0 + 2.0 ** -8)) == -1.0
    assert P.round_bf16(0.0) == 0.0
    assert P.round_bf16(255.0) == 255.0                            # 0b11111111: 8 significant bits fit
    assert P.round_bf16(257.0) == 256.0                            # 9 bits: tie between 256 (even) and 258
    assert P.round_bf16(259.0) == 260.0                            # tie between 258 (odd) and 260 (even)


def test_round_bf16_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(3)
    v = (torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 8)).numpy().astype(np.float32)
    # add exact ties: a bf16 value plus half its spacing
    base = (v[:2000].view(np.uint32) & 0xFFFF0000).view(np.float32)
    ties = (base.view(np.uint32) | 0x8000).view(np.float32)
    allv = np.concatenate([v, ties])
    np.testing.assert_array_equal(P.f64_to_bf16_bits(allv.astype(np.float64)), bf16_bits_of(allv))


# ------------------------------------------------------------------ RMSNorm and RoPE
def test_rms_norm_closed_form_and_scale_invariance():
    np.testing.assert_allclose(P.rms_norm([3.0, 4.0], eps=0.0), [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)],
                               rtol=1e-15)
    v = np.random.default_rng(1).standard_normal((5, 192))
    y = P.rms_norm(v, eps=0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(P.rms_norm(v * 1024.0, eps=0.0), y, rtol=1e-13)
    np.testing.assert_array_equal(P.rms_norm(np.zeros(8)), np.zeros(8))       # eps keeps zero at zero
    gamma = np.arange(1, 193, dtype=np.float64)
    np.testing.assert_allclose(P.rms_norm(v, gamma, eps=0.0), y * gamma, rtol=1e-15)
    # eps enters under the root: mean(v^2) = 1 for v = +-1, so the factor is 1 / sqrt(1 + eps)
    np.testing.assert_allclose(P.rms_norm(np.array([1.0, -1.0]), eps=0.25), [1 / math.sqrt(1.25), -1 / math.sqrt(1.25)],
                               rtol=1e-15)


def rope_complex(v, phi):
    """The rotation as complex multiplication of the pairs (v[2i] + i v[2i+1]) by e^{i phi}."""
    z = (v[..., 0::2] + 1j * v[..., 1::2]) * np.exp(1j * phi)
    out = np.empty(v.shape)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def test_rope_identity_quarter_turn_and_pairing():
    v = np.random.default_rng(2).standard_normal(64)
    np.testing.assert_array_equal(P.rope_interleaved(v, np.ones(32), np.zeros(32)), v)
    y = P.rope_interleaved(v, np.zeros(32), np.ones(32))           # 90 degrees: (a, b) -> (-b, a)
    np.testing.assert_array_equal(y[0::2], -v[1::2])
    np.testing.assert_array_equal(y[1::2], v[0::2])
    e0 = np.zeros(64)
    e0[0] = 1.0
    phi = 0.3
    y = P.rope_interleaved(e0, np.full(32, math.cos(phi)), np.full(32, math.sin(phi)))
    assert y[0] == pytest.approx(math.cos(phi)) and y[1] == pytest.approx(math.sin(phi))
    assert np.all(y[2:] == 0.0)                                    # dim 0 pairs with dim 1, not dim 32


def test_rope_equals_complex_rotation_and_keeps_pair_norms():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((7, 64))
    phi = rng.uniform(0, 2 * math.pi, (7, 32))
    y = P.rope_interleaved(v, np.cos(phi), np.sin(phi))
    np.testing.assert_allclose(y, rope_complex(v, phi), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y[:, 0::2] ** 2 + y[:, 1::2] ** 2, v[:, 0::2] ** 2 + v[:, 1::2] ** 2, rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal(64), rng.standard_normal(64)
    theta = 10000.0 ** (-np.arange(32) * 2.0 / 64.0)

    def rot(v, p):
        return P.rope_interleaved(v, np.cos(p * theta), np.sin(p * theta))

    s = np.dot(rot(a, 1000), rot(b, 990))
    for shift in (1, 37, 5000):
        assert np.dot(rot(a, 1000 + shift), rot(b, 990 + shift)) == pytest.approx(s, rel=1e-9, abs=1e-9)
    assert abs(np.dot(rot(a, 1000), rot(b, 980)) - s) > 1e-3     # another distance gives another score


# ------------------------------------------------------------------ the whole prolog
def selection_inputs(seed=6, T=3, H=2):
    """hidden 576, q_lora = H * 192: wq_a picks x[:q_lora], wq_b and wkv are identities."""
    rng = np.random.default_rng(seed)
    hidden, q_lora = 576, H * 192
    x = bf16_bits_of(rng.standard_normal((T, hidden)))
    wq_a = np.zeros((hidden, q_lora), np.float32)
    wq_a[:q_lora, :q_lora] = np.eye(q_lora)
    phi = rng.uniform(0, 2 * math.pi, (T, 32))
    return dict(x=x, wq_a=bf16_bits_of(wq_a), gamma_cq=bf16_bits_of(rng.uniform(0.5, 1.5, q_lora)),
                wq_b=bf16_bits_of(np.eye(q_lora)), w_uk=bf16_bits_of(rng.standard_normal((H, 128, 512)) / 11),
                wkv=bf16_bits_of(np.eye(576)), gamma_ckv=bf16_bits_of(rng.uniform(0.5, 1.5, 576)),
                cos=np.cos(phi).astype(np.float32), sin=np.sin(phi).astype(np.float32)), phi


def test_closed_form_with_selection_weights():
    """With wq_b = I the first RMSNorm's factor cancels in the per-head second
    one, leaving q_h = RMSNorm((gamma_cq * x)[head h's 192]); with wkv = I the
    key row is RMSNorm(x) * gamma_ckv.  eps = 0 keeps both exact."""
    inp, phi = selection_inputs()
    out = P.forward(inp, round_intermediates=False, eps=0.0)
    x = P.bf16_to_f64(inp["x"])
    g_cq, g_ckv = P.bf16_to_f64(inp["gamma_cq"]), P.bf16_to_f64(inp["gamma_ckv"])
    w_uk = P.bf16_to_f64(inp["w_uk"])
    phi32 = np.arctan2(inp["sin"].astype(np.float64), inp["cos"].astype(np.float64))
    radius = np.hypot(inp["sin"].astype(np.float64), inp["cos"].astype(np.float64))
    for t in range(3):
        for h in range(2):
            v = (g_cq * x[t, :384])[192 * h:192 * (h + 1)]
            qh = v / math.sqrt(float(np.dot(v, v)) / 192)
            np.testing.assert_allclose(out["q_rope"][t, h], rope_complex(qh[128:], phi32[t]) * _pair_radius(radius[t]),
                                       rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(out["q_nope"][t, h], qh[:128] @ w_uk[h], rtol=1e-11, atol=1e-12)
        k = x[t] / math.sqrt(float(np.dot(x[t], x[t])) / 576) * g_ckv
        np.testing.assert_allclose(out["k_nope_exact"][t], k[:512], rtol=1e-13)
        np.testing.assert_allclose(out["k_rope_exact"][t], rope_complex(k[512:], phi32[t]) * _pair_radius(radius[t]),
                                   rtol=1e-12, atol=1e-12)


def _pair_radius(r):
    """The fp32 cos / sin inputs are a rotation times |e^{i phi}| = hypot(cos, sin), which is 1 only up to fp32 rounding."""
    return np.repeat(r, 2)


def test_head_permutation_permutes_outputs():
    inp = workloads.make_prolog_inputs(T=4, seed=7, hidden=64, q_lora=32, n_heads=4, num_blocks=1)
    out = P.forward(inp)
    perm = np.array([2, 0, 3, 1])
    wq_b = inp["wq_b"].reshape(32, 4, 192)[:, perm].reshape(32, 4 * 192)
    out2 = P.forward(dict(inp, wq_b=wq_b, w_uk=inp["w_uk"][perm]))
    np.testing.assert_array_equal(out2["q_nope"], out["q_nope"][:, perm])
    np.testing.assert_array_equal(out2["q_rope"], out["q_rope"][:, perm])
    np.testing.assert_array_equal(out2["k_nope"], out["k_nope"])


def test_absorbed_query_scores_equal_up_projected_keys():
    """Absorption: q_abs[h] . c = q_nope[h] . (w_uk[h] @ c) for any latent c."""
    inp = workloads.make_prolog_inputs(T=3, seed=8, hidden=64, q_lora=32, n_heads=3, num_blocks=1)
    out = P.forward(inp)
    c = np.random.default_rng(9).standard_normal((5, 512))
    w_uk = P.bf16_to_f64(inp["w_uk"])
    for h in range(3):
        lhs = out["q_nope"][:, h] @ c.T
        rhs = out["q_head"][:, h, :128] @ (w_uk[h] @ c.T)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-10)


def test_zero_row_scaled_row_and_storage_points():
    inp = workloads.make_prolog_inputs(T=4, seed=10, hidden=64, q_lora=32, n_heads=2, num_blocks=1)
    out = P.forward(inp)
    assert np.all(out["q_nope"][1] == 0) and np.all(out["q_rope"][1] == 0) and np.all(out["k_nope"][1] == 0)
    # a row times 2^10 (exact in bf16): with eps = 0 every output is the unscaled row's
    x = inp["x"].copy()
    x[3] = bf16_bits_of(P.bf16_to_f64(x[0]) * 1024.0)
    with np.errstate(invalid="ignore"):                            # row 1 is zero: 0 / 0 without eps
        e = P.forward(dict(inp, x=x, cos=np.repeat(inp["cos"][:1], 4, 0), sin=np.repeat(inp["sin"][:1], 4, 0)),
                      eps=0.0)
    np.testing.assert_allclose(e["q_nope"][3], e["q_nope"][0], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(e["k_nope"][3], e["k_nope"][0])
    # storage points: c^Q and the pre-absorption query are bf16 values; the exact run differs by rounding only
    assert np.array_equal(P.round_bf16(out["c_q"]), out["c_q"])
    assert np.array_equal(P.round_bf16(out["q_head"][..., :128]), out["q_head"][..., :128])
    ex = P.forward(inp, round_intermediates=False)
    rms = np.sqrt(np.mean(ex["q_nope"] ** 2, axis=-1, keepdims=True)) + 1e-30
    assert np.max(np.abs(out["q_nope"] - ex["q_nope"]) / rms) < 2.0 ** -5
    assert np.max(np.abs(out["q_nope"] - ex["q_nope"])) > 0       # the rounding points are really there


def test_cache_rows_are_the_rounded_key_and_go_through_the_writer():
    inp = workloads.prolog_tiny()
    out, (kn, kr, ks, bad) = P.forward_with_cache(inp)
    np.testing.assert_array_equal(out["k_nope"], P.f64_to_bf16_bits(out["k_nope_exact"]))
    np.testing.assert_array_equal(out["k_rope"], P.f64_to_bf16_bits(out["k_rope_exact"]))
    kn2, kr2, _, _ = cache_write(out["k_nope"], out["k_rope"], inp["cache_index"], inp["kv_nope"], inp["kv_rope"])
    np.testing.assert_array_equal(kn, kn2)
    np.testing.assert_array_equal(kr, kr2)
    assert bad == 0
    written = inp["cache_index"][inp["cache_index"] >= 0]
    untouched = np.setdiff1d(np.arange(kn.shape[0]), written)
    np.testing.assert_array_equal(kn[untouched], inp["kv_nope"][untouched])
    t = int(np.nonzero(inp["cache_index"] >= 0)[0][0])
    np.testing.assert_array_equal(kn[inp["cache_index"][t]], out["k_nope"][t])
