"""Pins of the paged cache writer oracle ("DeepSeek V3/V2 Sparse Flash Attention
with Quantization", sections on the operator spec, inputs/outputs and the INT8
quantisation rule; "NPU DeepSeek-V4 PyPTO fused-operator optimization",
section MlaProlog): bf16 rows land bit for bit, INT8 codes and scales match
closed forms, round half to even, the rounding bound, and an independent torch
implementation of the same rule.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def f32_to_bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bits (test-side helper for building inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def empty_cache(rows, int8):
    kn = np.full((rows, 512), 7, dtype=np.int8) if int8 else np.full((rows, 512), 0x3F80, dtype=np.uint16)
    kr = np.full((rows, 64), 0x4000, dtype=np.uint16)
    ks = np.full((rows, 4), 9.0, dtype=np.float32) if int8 else None
    return kn, kr, ks


def test_bf16_rows_land_bit_for_bit_and_others_are_untouched():
    rng = np.random.default_rng(0)
    T, rows = 6, 40
    kn_new = f32_to_bf16_bits(rng.standard_normal((T, 512)))
    kr_new = f32_to_bf16_bits(rng.standard_normal((T, 64)))
    idx = np.array([3, 39, -1, 17, 40, 0], dtype=np.int64)    # -1 skipped, 40 out of range
    kn, kr, _ = empty_cache(rows, False)
    on, orr, _, bad = oracle.cache_write(kn_new, kr_new, idx, kn, kr)
    assert bad == 1
    for t, r in enumerate(idx):
        if 0 <= r < rows:
            np.testing.assert_array_equal(on[r], kn_new[t])
            np.testing.assert_array_equal(orr[r], kr_new[t])
    untouched = np.setdiff1d(np.arange(rows), idx[(idx >= 0) & (idx < rows)])
    assert (on[untouched] == 0x3F80).all() and (orr[untouched] == 0x4000).all()


def test_int8_exact_multiples_of_the_scale():
    """Group values k * 2^-3 with one |k| = 127: scale is exactly 2^-3 and every
    code is exactly k."""
    rng = np.random.default_rng(1)
    k = rng.integers(-127, 128, size=(1, 512)).astype(np.int64)
    for g in range(4):
        k[0, g * 128 + 5 + g] = 127 if g % 2 == 0 else -127
    x = (k * 2.0 ** -3).astype(np.float32)
    kn, kr, ks = empty_cache(2, True)
    on, _, os_, _ = oracle.cache_write(f32_to_bf16_bits(x), np.zeros((1, 64), np.uint16), np.array([1]), kn, kr, ks)
    np.testing.assert_array_equal(on[1].astype(np.int64), k[0])
    np.testing.assert_array_equal(os_[1], np.full(4, 2.0 ** -3, dtype=np.float32))
    assert (on[0] == 7).all() and (os_[0] == 9.0).all()


def test_int8_rounds_half_to_even_and_zero_groups_get_scale_one():
    x = np.zeros((1, 512), dtype=np.float32)
    x[0, 0] = 127.0                                                # group 0: scale exactly 1
    x[0, 1:9] = [0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5]
    # group 1 stays all zero
    x[0, 256] = -127.0                                             # group 2: scale 1, negative extreme
    x[0, 384] = 2.0 ** -20                                         # group 3: tiny, scale = 2^-20 / 127
    kn, kr, ks = empty_cache(1, True)
    on, _, os_, _ = oracle.cache_write(f32_to_bf16_bits(x), np.zeros((1, 64), np.uint16), np.array([0]), kn, kr, ks)
    np.testing.assert_array_equal(on[0, :9], [127, 0, 2, 2, 0, -2, -2, 4, 126])
    assert os_[0, 0] == 1.0 and os_[0, 1] == 1.0 and (on[0, 128:256] == 0).all()
    assert on[0, 256] == -127 and os_[0, 2] == 1.0
    assert on[0, 384] == 127 and os_[0, 3] == np.float32(np.float32(2.0 ** -20) / np.float32(127.0))


@pytest.mark.parametrize("sigma", [1e-3, 1.0, 1e3])
def test_int8_rounding_bound_and_extremes(sigma):
    rng = np.random.default_rng(2)
    T = 16
    x = bf16_to_f32(f32_to_bf16_bits(rng.standard_normal((T, 512)) * sigma))
    kn, kr, ks = empty_cache(T, True)
    on, _, os_, _ = oracle.cache_write(f32_to_bf16_bits(x), np.zeros((T, 64), np.uint16), np.arange(T), kn, kr, ks)
    grp = x.reshape(T, 4, 128).astype(np.float64)
    q = on.reshape(T, 4, 128).astype(np.float64)
    s = os_.astype(np.float64)[..., None]
    # x / scale is rounded once in fp32 (|x / scale| <= 127, so by <= 127 * 2^-24),
    # then to the nearest integer: |code * scale - x| <= scale * (1/2 + 2^-16)
    assert np.all(np.abs(q * s - grp) <= s * (0.5 + 2.0 ** -16))
    am = np.abs(grp).argmax(axis=-1)
    ext = np.take_along_axis(q, am[..., None], -1)[..., 0]
    np.testing.assert_array_equal(np.abs(ext), 127)
    np.testing.assert_array_equal(np.sign(ext), np.sign(np.take_along_axis(grp, am[..., None], -1)[..., 0]))
    assert q.min() >= -127 and q.max() <= 127


def test_int8_equals_an_independent_torch_quantiser():
    """workloads.quantize_int8_groups (torch ops, written separately) on the same
    bf16-valued inputs gives the same codes and scales."""
    rng = np.random.default_rng(3)
    T = 32
    x = bf16_to_f32(f32_to_bf16_bits(rng.standard_normal((T, 512)) * rng.uniform(0.01, 10, size=(T, 1))))
    x[5, 128:256] = 0.0
    q_ref, s_ref = workloads.quantize_int8_groups(torch.from_numpy(x.copy()))
    kn, kr, ks = empty_cache(T, True)
    on, _, os_, _ = oracle.cache_write(f32_to_bf16_bits(x), np.zeros((T, 64), np.uint16), np.arange(T), kn, kr, ks)
    np.testing.assert_array_equal(on, q_ref)
    np.testing.assert_array_equal(os_, s_ref)


def test_rope_rows_are_copied_in_both_modes():
    rng = np.random.default_rng(4)
    kr_new = f32_to_bf16_bits(rng.standard_normal((3, 64)))
    for int8 in (False, True):
        kn, kr, ks = empty_cache(5, int8)
        kn_new = np.zeros((3, 512), np.uint16)
        _, orr, _, _ = oracle.cache_write(kn_new, kr_new, np.array([4, 2, 0]), kn, kr, ks)
        np.testing.assert_array_equal(orr[[4, 2, 0]], kr_new)
        assert (orr[[1, 3]] == 0x4000).all()
