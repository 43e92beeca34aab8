"""Pins of the oracle's building blocks against closed forms, library routines,
brute force and published known-answer vectors (CPU only)."""
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- FP16 codec

def test_half_to_float_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_float_to_half_round_to_nearest_even_matches_numpy():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.05),
        rng.standard_normal(5000).astype(np.float32) * np.float32(3000.0),
        (rng.random(5000).astype(np.float32) * np.float32(1e-4)),     # subnormal half range
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11], dtype=np.float32),
    ])
    # exact ties between two binary16 neighbours: k + 0.5 quanta
    ties = ((np.arange(1024, 2048, 7, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10))
    vals = np.concatenate([vals, ties, -ties])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- matvec

def test_matvec_integer_inputs_exact():
    rng = np.random.default_rng(1)
    W = rng.integers(-3, 4, size=(37, 53)).astype(np.float16)
    x = rng.integers(-5, 6, size=53).astype(np.float32)
    exact = W.astype(np.int64) @ x.astype(np.int64)
    assert np.array_equal(oracle.matvec(W, x), exact.astype(np.float32))


def test_matvec_rectangular_orientation():
    # y_r = sum_k W[r, k] x_k: a one-hot x picks out column k of W (row-major [rows, cols]).
    W = (np.arange(5 * 9, dtype=np.float32).reshape(5, 9) / 64).astype(np.float16)
    for k in (0, 4, 8):
        x = np.zeros(9, dtype=np.float32)
        x[k] = 1.0
        assert np.array_equal(oracle.matvec(W, x), W[:, k].astype(np.float32))


def test_matvec_within_fp32_sum_bound_of_fp64_brute_force():
    rng = np.random.default_rng(2)
    for n, k in ((3, 7), (16, 256), (5, 4099)):
        W = (rng.standard_normal((n, k)) * 0.02).astype(np.float16)
        x = rng.standard_normal(k).astype(np.float32)
        y = oracle.matvec(W, x).astype(np.float64)
        Wd, xd = W.astype(np.float64), x.astype(np.float64)
        ref = np.array([sum(Wd[r, j] * xd[j] for j in range(k)) for r in range(n)])
        bound = (k + 1) * 2.0 ** -24 * (np.abs(Wd) @ np.abs(xd))
        assert np.all(np.abs(y - ref) <= bound)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_forms():
    ones = np.ones(64, dtype=np.float16)
    for c in (0.5, 3.0, -2.0):
        out = oracle.rmsnorm(np.full(64, c, np.float32), ones, 1e-5)
        np.testing.assert_allclose(out, c / math.sqrt(c * c + 1e-5), rtol=1e-6)
    pm = np.where(np.arange(64) % 3 == 0, 1.0, -1.0).astype(np.float32)
    np.testing.assert_allclose(oracle.rmsnorm(pm, ones, 1e-5), pm / math.sqrt(1 + 1e-5), rtol=1e-6)
    # eps only matters against the mean square: x = 0 gives 0
    assert np.all(oracle.rmsnorm(np.zeros(8, np.float32), ones[:8], 1e-5) == 0)


def test_rmsnorm_unit_rms_scale_invariance_and_gain():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(1024).astype(np.float32) * 7
    g = (1 + 0.1 * rng.standard_normal(1024)).astype(np.float16)
    ones = np.ones(1024, dtype=np.float16)
    y = oracle.rmsnorm(x, ones, 0.0)
    assert abs(float(np.mean(y.astype(np.float64) ** 2)) - 1.0) < 1e-5
    np.testing.assert_allclose(oracle.rmsnorm(np.float32(1000) * x, ones, 1e-5), y, rtol=2e-6, atol=1e-7)
    yg = oracle.rmsnorm(x, g, 0.0)
    np.testing.assert_array_equal(yg, y * g.astype(np.float32))


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(128).astype(np.float32)
    assert np.array_equal(oracle.rope(v, 0, 10000.0), v)


def test_rope_pairs_and_frequencies_closed_form():
    hd, base = 64, 10000.0
    for i in (0, 5, 31):
        for pos in (1, 17, 1000):
            v = np.zeros(hd, np.float32)
            v[i] = 1.0
            out = oracle.rope(v, pos, base)
            ang = pos * base ** (-2.0 * i / hd)
            expect = np.zeros(hd)
            expect[i] = math.cos(ang)
            expect[i + hd // 2] = math.sin(ang)   # rotate-half partner of element i
            np.testing.assert_allclose(out, expect, atol=2e-7)


def test_rope_preserves_pair_norms_and_relative_positions():
    rng = np.random.default_rng(5)
    hd = 128
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    for pos in (3, 511, 32000):
        r = oracle.rope(q, pos, 10000.0).astype(np.float64)
        before = q[:64].astype(np.float64) ** 2 + q[64:].astype(np.float64) ** 2
        after = r[:64] ** 2 + r[64:] ** 2
        np.testing.assert_allclose(after, before, rtol=1e-6)
    # <R_m q, R_n k> depends only on m - n
    a = np.dot(oracle.rope(q, 40, 10000.0).astype(np.float64), oracle.rope(k, 10, 10000.0))
    b = np.dot(oracle.rope(q, 30, 10000.0).astype(np.float64), k.astype(np.float64))
    assert abs(a - b) < 1e-4


# ---------------------------------------------------------------- attention

def _kv(rng, ctx, hd):
    return ((rng.standard_normal((ctx, hd)) * 0.5).astype(np.float16),
            rng.standard_normal((ctx, hd)).astype(np.float16))


def test_attention_single_position_returns_v_exactly():
    rng = np.random.default_rng(6)
    K, V = _kv(rng, 1, 64)
    q = rng.standard_normal(64).astype(np.float32)
    out, p = oracle.attend_head(q, K, V, 0.125)
    assert p[0] == 1.0
    assert np.array_equal(out, V[0].astype(np.float32))


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(7)
    ctx, hd = 50, 64
    K = np.tile(rng.standard_normal((1, hd)).astype(np.float16), (ctx, 1))
    V = rng.standard_normal((ctx, hd)).astype(np.float16)
    q = rng.standard_normal(hd).astype(np.float32)
    out, p = oracle.attend_head(q, K, V, 0.125)
    np.testing.assert_allclose(p, 1.0 / ctx, rtol=1e-6)
    np.testing.assert_allclose(out, V.astype(np.float64).mean(axis=0), atol=2e-6)


def test_attention_probabilities_match_library_softmax_and_scale():
    rng = np.random.default_rng(8)
    ctx, hd = 300, 128
    K, V = _kv(rng, ctx, hd)
    q = rng.standard_normal(hd).astype(np.float32)
    scale = np.float32(1.0) / np.sqrt(np.float32(hd))
    out, p = oracle.attend_head(q, K, V, float(scale))
    assert abs(float(np.sum(p, dtype=np.float64)) - 1.0) < 1e-6
    s = (K.astype(np.float64) @ q.astype(np.float64)) * float(scale)
    np.testing.assert_allclose(p, special.softmax(s), rtol=2e-5, atol=1e-9)
    np.testing.assert_allclose(out, special.softmax(s) @ V.astype(np.float64), atol=2e-5)
    # the probability ratio of two keys is exp(scale * (q.k1 - q.k2))
    i, j = int(np.argmax(p)), int(np.argmin(p))
    np.testing.assert_allclose(math.log(p[i] / p[j]), (s[i] - s[j]), rtol=1e-4)


# ---------------------------------------------------------------- SiLU

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    # silu(ln 3) = ln 3 * sigmoid(ln 3) = 0.75 ln 3
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-6
    for z in (0.3, 1.7, 5.0, 11.0):
        assert abs((oracle.silu(z) - oracle.silu(-z)) - z) < 2e-6 * max(1.0, z)
    assert abs(oracle.silu(30.0) - 30.0) < 1e-5
    assert abs(oracle.silu(-30.0)) < 1e-10


# ---------------------------------------------------------------- Philox / Gumbel / sampling

def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if len(line) == 10:
                rows.append([int(v, 16) for v in line])
    assert len(rows) == 3
    return rows


def test_philox_known_answer_vectors():
    for r in _kat_rows():
        assert oracle.philox4x32_10(r[0:4], r[4:6]) == r[6:10]


def test_gumbel_noise_follows_standard_gumbel_cdf():
    g = np.array([oracle.gumbel(99, pos, i) for pos in range(40) for i in range(500)])
    assert np.all(np.isfinite(g))
    ks = stats.kstest(g, "gumbel_r")
    assert ks.pvalue > 1e-3
    assert abs(g.mean() - np.euler_gamma) < 0.03


def test_gumbel_noise_depends_on_seed_position_and_index():
    a = oracle.gumbel(1, 10, 5)
    assert a != oracle.gumbel(2, 10, 5) and a != oracle.gumbel(1, 11, 5) and a != oracle.gumbel(1, 10, 6)
    assert a == oracle.gumbel(1, 10, 5)


def test_sampling_distribution_is_softmax_over_top_k():
    logits = np.array([1.0, 0.2, -0.5, 0.9, 2.0, -1.0, 0.0, 0.5], dtype=np.float32)
    T, k, n = 0.8, 5, 60000
    counts = np.zeros(8)
    for pos in range(n):
        counts[oracle.sample(logits, T, k, 4242, pos)] += 1
    top = np.argsort(-logits, kind="stable")[:k]
    p = np.zeros(8)
    p[top] = special.softmax(logits[top].astype(np.float64) / T)
    assert np.all(counts[p == 0] == 0)
    chi = stats.chisquare(counts[top], n * p[top])
    assert chi.pvalue > 1e-3


def test_sampling_degenerate_cases_reduce_to_greedy():
    rng = np.random.default_rng(9)
    for trial in range(20):
        lg = rng.standard_normal(1000).astype(np.float32)
        greedy = oracle.sample(lg, 0.0, 0, 1, trial)
        assert greedy == int(np.argmax(lg))
        assert oracle.sample(lg, 0.7, 1, 123, trial) == greedy           # top-k = 1
        assert oracle.sample(lg, 1e-6, 0, 123, trial) == greedy          # T -> 0
    lg = np.zeros(16, np.float32)
    lg[[3, 9]] = 1.0
    assert oracle.sample(lg, 0.0, 0, 0, 0) == 3                           # lower index wins ties


def test_sampling_top_k_ties_at_boundary_take_lower_index():
    lg = np.array([0.0, 5.0, 1.0, 1.0, 1.0, -3.0], dtype=np.float32)
    seen = {oracle.sample(lg, 50.0, 3, 77, pos) for pos in range(400)}
    assert seen <= {1, 2, 3} and {2, 3} <= seen
