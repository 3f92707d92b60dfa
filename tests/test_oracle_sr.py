"""Pins of the oracle's stochastic rounding of the bf16 state ([M2] 评论区精华:
stochastic rounding for quantised models): the Philox4x32-10 generator against its
published known-answer vectors, and the rounding rule against its defining
properties (exact mean over all random inputs, neighbours only, symmetry, agreement
with round-to-nearest where that is forced)."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w = [int(t, 16) for t in line.split()]
        rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,out", _kat())
def test_philox_known_answers(ctr, key, out):
    assert oracle.philox4x32_10(ctr, key) == out


def test_philox_counter_and_key_change_output():
    base = oracle.philox4x32_10([1, 2, 3, 4], [5, 6])
    for i in range(4):
        c = [1, 2, 3, 4]
        c[i] ^= 1
        assert oracle.philox4x32_10(c, [5, 6]) != base
    assert oracle.philox4x32_10([1, 2, 3, 4], [5, 7]) != base


def test_sr_bits_layout():
    # element e draws half (e % 2) of word (e % 8) / 2 of the block at counter e / 8
    seed, off = 0x0123456789ABCDEF, 0xFEDCBA9876543210
    for e in (0, 1, 5, 7, 8, 23, (1 << 35) + 6):
        g = e // 8
        w = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, off & 0xFFFFFFFF, off >> 32],
                                 [seed & 0xFFFFFFFF, seed >> 32])
        word = w[(e % 8) // 2]
        want = (word >> (16 * (e % 2))) & 0xFFFF
        assert oracle.sr_bits(seed, off, e) == want


def _bf16_neighbours(v):
    """The bf16 values next to float32 v toward and away from zero, via torch's
    bfloat16 type (truncation of the float32 bit pattern)."""
    f = np.float32(v)
    bits = np.array([f], dtype=np.float32).view(np.uint32)[0]
    lo = np.array([bits & 0xFFFF0000], dtype=np.uint32).view(np.float32)[0]
    hi = np.array([(bits & 0xFFFF0000) + 0x10000], dtype=np.uint32).view(np.float32)[0]
    return float(lo), float(hi)


@pytest.mark.parametrize("v", [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -10, -0.3, 3.14159,
                               -1.2345e-3, 7.0e20, 1.0e-39, -2.5e-41])
def test_sr_mean_over_all_bits_is_exact(v):
    v32 = float(np.float32(v))
    vals = np.array([oracle.round_bf16_sr(v32, r) for r in range(65536)])
    lo, hi = _bf16_neighbours(v32)
    assert set(np.unique(vals)) <= {lo, hi}
    # the up-count is exactly 2^16 times the dropped fraction: mean equals v
    assert vals.sum() / 65536.0 == pytest.approx(v32, rel=0, abs=0)


def test_sr_sign_symmetry_and_fixed_points():
    rng = np.random.default_rng(3)
    for v in rng.standard_normal(200):
        r = int(rng.integers(0, 65536))
        assert oracle.round_bf16_sr(-v, r) == -oracle.round_bf16_sr(v, r)
    # bf16 values and specials pass through for every r
    for v in (0.0, -0.0, 1.0, -0.5, 2.0 ** -133, float(torch.tensor(0.7).bfloat16())):
        for r in (0, 1, 32767, 65535):
            assert oracle.round_bf16_sr(v, r) == v
    assert np.isnan(oracle.round_bf16_sr(float("nan"), 5))
    assert oracle.round_bf16_sr(float("inf"), 65535) == float("inf")


def test_sr_extreme_bits_are_truncation_and_round_up():
    # r = 0 never rounds away from zero (unless v is a bf16 value already); r = 2^16 - 1
    # rounds away whenever a fraction is dropped
    rng = np.random.default_rng(4)
    for v in rng.standard_normal(300) * 10.0 ** rng.integers(-20, 20, 300):
        v32 = float(np.float32(v))
        lo, hi = _bf16_neighbours(v32)
        assert oracle.round_bf16_sr(v32, 0) == lo
        want = lo if lo == v32 else hi
        assert oracle.round_bf16_sr(v32, 65535) == want


def test_round_slots_sr_matches_per_element_rule():
    rng = np.random.default_rng(5)
    pool = rng.standard_normal((5, 3, 16))
    ref = pool.copy()
    oracle.round_slots_sr(pool, [3, -1, 1], seed=77, offset=9)
    for s in range(5):
        for j in range(48):
            e = s * 48 + j
            v = ref[s].reshape(-1)[j]
            want = oracle.round_bf16_sr(v, oracle.sr_bits(77, 9, e)) if s in (1, 3) else v
            assert pool[s].reshape(-1)[j] == want


def test_sr_is_unbiased_on_random_values_where_nearest_is_not_needed():
    # averaged over seeds, SR of a fixed value converges to it (error ~ ulp / sqrt(T)),
    # while a single round-to-nearest keeps an error of ~ ulp / 4 on average
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(512) * 3.0).astype(np.float32).astype(np.float64)
    pool = np.repeat(v[None, :], 1, axis=0)
    T = 256
    acc = np.zeros_like(v)
    for t in range(T):
        p = pool.copy()
        oracle.round_slots_sr(p, [0], seed=11, offset=t)
        acc += p[0]
    mean = acc / T
    ulp = np.array([abs(_bf16_neighbours(x)[1] - _bf16_neighbours(x)[0]) for x in v])
    rne = np.array([oracle.round_bf16(x) for x in v])
    err_sr = np.mean(np.abs(mean - v) / ulp)
    err_rne = np.mean(np.abs(rne - v) / ulp)
    assert err_rne > 0.2
    assert err_sr < 0.05
