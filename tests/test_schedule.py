"""Host-side scheduling half of section 2.A (no GPU): the oracle against brute force and
closed forms, then the C-ABI functions against the oracle."""
import math

import numpy as np
import pytest

import adaln_layernorm_modulate_gb300 as A
import synth
from oracle import bucket as obucket
from oracle import schedule as osched

M_MEM, M_COMP = synth.BUCKET_M_MEM, synth.BUCKET_M_COMP


# ---- bucket size with a real exponent ----------------------------------------------------
def brute_force_half(S, M_mem, M_comp, p2):
    """p = p2 / 2 with S a perfect square: S^p = isqrt(S)^p2, an exact integer."""
    r = math.isqrt(S)
    assert r * r == S
    sp = r ** p2
    return max(1, min(M_mem // S, M_comp // sp))


@pytest.mark.parametrize("S", [256, 1024, 4096, 16384, 65536, 9, 49])
@pytest.mark.parametrize("p2", [3, 5, 7])
def test_half_integer_exponents_against_brute_force(S, p2):
    for M_mem, M_comp in [(M_MEM, M_COMP), (10 ** 9, 10 ** 12), (7, 3 ** 20 + 1)]:
        want = brute_force_half(S, M_mem, M_comp, p2)
        got, near = osched.bucket_batch_real(S, M_mem, M_comp, p2 / 2)
        assert got == want
        if not near:
            assert A.adaln_bucket_batch_real(S, M_mem, M_comp, p2 / 2) == want


def test_integral_exponents_take_the_exact_rule():
    for S in (1, 2, 256, 32760, 75600, 10 ** 6):
        for p in (1, 2, 3, 7):
            want = obucket.bucket_batch(S, M_MEM, M_COMP, p)
            assert osched.bucket_batch_real(S, M_MEM, M_COMP, float(p)) == (want, False)
            assert A.adaln_bucket_batch_real(S, M_MEM, M_COMP, float(p)) == want


def test_real_exponents_match_the_oracle():
    rng = np.random.default_rng(11)
    checked = 0
    for _ in range(400):
        S = int(rng.integers(1, 200000))
        p = float(rng.uniform(0.5, 3.5))
        M_mem = int(rng.integers(1, 10 ** 7))
        M_comp = int(rng.integers(1, 10 ** 13))
        want, near = osched.bucket_batch_real(S, M_mem, M_comp, p)
        if near:
            continue
        assert A.adaln_bucket_batch_real(S, M_mem, M_comp, p) == want, (S, M_mem, M_comp, p)
        checked += 1
    assert checked > 390


def test_real_exponent_rejects_bad_arguments():
    for args in [(0, 1, 1, 2.0), (1, 0, 1, 2.0), (1, 1, 0, 2.0), (1, 1, 1, 0.0), (1, 1, 1, -1.5),
                 (1, 1, 1, float("nan")), (1, 1, 1, float("inf"))]:
        assert A.adaln_bucket_batch_real(*args) == -1


# ---- Shape-Benchmarking fit ---------------------------------------------------------------
def samples(seed, a, b, p, n=60, noise=0.0):
    rng = np.random.default_rng(seed)
    B = rng.integers(1, 128, n)
    S = rng.choice(np.array(synth.BUCKET_S), n)
    t = a + b * B * S.astype(np.float64) ** p
    if noise:
        t = t * (1 + noise * rng.standard_normal(n))
    return B, S, t


def test_oracle_fit_recovers_noise_free_parameters():
    a, b, p = 0.37, 3e-9, 1.83
    B, S, t = samples(1, a, b, p)
    f = osched.fit_step_cost(B, S, t, 1.0, 3.0, a + b * 123456.0)
    assert abs(f["p"] - p) < 1e-8
    assert abs(f["a"] - a) <= 1e-6 * a and abs(f["b"] - b) <= 1e-6 * b
    assert f["M_comp"] in (123455.0, 123456.0)  # floor of a value equal to 123456 up to rounding


def test_oracle_fit_agrees_with_a_generic_solver_on_noisy_data():
    opt = pytest.importorskip("scipy.optimize")
    B, S, t = samples(2, 0.5, 2e-9, 2.1, noise=0.02)
    f = osched.fit_step_cost(B, S, t, 1.0, 3.0, 1.0)
    model = lambda X, a, b9, p: a + b9 * 1e-9 * X[0] * X[1] ** p  # b in units of 1e-9
    (a, b9, p), _ = opt.curve_fit(model, np.stack([B, S.astype(np.float64)]), t, p0=[0.4, 1.0, 2.0],
                                  maxfev=20000)
    assert abs(f["p"] - p) < 1e-5


@pytest.mark.parametrize("seed,params,noise", [(3, (0.37, 3e-9, 1.83), 0.0), (4, (0.5, 2e-9, 2.1), 0.02),
                                               (5, (1.0, 1e-7, 1.2), 0.05)])
def test_library_fit_matches_the_oracle(seed, params, noise):
    B, S, t = samples(seed, *params, noise=noise)
    budget = params[0] + params[1] * 5e7
    want = osched.fit_step_cost(B, S, t, 1.0, 3.0, budget)
    got = A.adaln_fit_step_cost(B, S, t, 1.0, 3.0, budget)
    assert abs(got["p"] - want["p"]) < 1e-6
    assert abs(got["a"] - want["a"]) <= 1e-5 * abs(want["a"]) + 1e-12
    assert abs(got["b"] - want["b"]) <= 1e-5 * abs(want["b"])
    # As good a minimum as the oracle's, up to the rounding noise of the data.
    assert got["rms"] <= want["rms"] * (1 + 1e-6) + 1e-12 * float(np.sqrt(np.mean(t * t)))
    assert abs(got["M_comp"] - want["M_comp"]) <= 1e-4 * want["M_comp"] + 1


def test_fit_rejects_bad_arguments():
    with pytest.raises(A.AdalnError):
        A.adaln_fit_step_cost([1, 2], [3, 4], [0.1, 0.2])
    with pytest.raises(A.AdalnError):
        A.adaln_fit_step_cost([1, 2, 3], [3, 0, 4], [0.1, 0.2, 0.3])
    with pytest.raises(A.AdalnError):
        A.adaln_fit_step_cost([1, 2, 3], [3, 2, 4], [0.1, 0.2, 0.3], p_lo=2.0, p_hi=1.0)


# ---- compute-load imbalance ---------------------------------------------------------------
def test_load_cv_hand_example():
    # Buckets 2 and 4, p = 2, M_mem = 8: 5 samples of length <= 2, 3 of length 3..4.
    lengths = [1, 2, 2, 1, 2, 3, 4, 4]
    # Equal-token: sizes 4 and 2 -> batches (2: 4 samples, 1 sample), (4: 2, 1)
    # costs 4*4 = 16, 1*4 = 4, 2*16 = 32, 1*16 = 16: mean 17, variance 99.
    want_cv = math.sqrt(99.0) / 17.0
    for got in (osched.bucket_load_cv(lengths, [2, 4], 8, 10 ** 6, 2.0, 0),
                A.adaln_bucket_load_cv(lengths, [2, 4], 8, 10 ** 6, 2.0, 0)):
        assert got["batches"] == 4 and got["mean"] == 17.0
        assert abs(got["cv"] - want_cv) < 1e-12
    # Dual constraint with M_comp = 16: sizes min(4, 16/4) = 4 and min(2, 16/16) = 1 ->
    # costs 16, 4, 16, 16, 16: mean 13.6, variance (4*2.4^2 + 9.6^2) / 5 = 23.04.
    want_cv = math.sqrt(23.04) / 13.6
    for got in (osched.bucket_load_cv(lengths, [2, 4], 8, 16, 2.0, 1),
                A.adaln_bucket_load_cv(lengths, [2, 4], 8, 16, 2.0, 1)):
        assert got["batches"] == 5 and abs(got["mean"] - 13.6) < 1e-12
        assert abs(got["cv"] - want_cv) < 1e-12


def mixed_lengths(seed, n):
    """Seeded log-uniform lengths between 100 and 75,600 tokens (a mixed-resolution mix)."""
    rng = np.random.default_rng(seed)
    return np.exp(rng.uniform(math.log(100), math.log(75600), n)).astype(np.int64)


@pytest.mark.parametrize("rule", [0, 1])
@pytest.mark.parametrize("p", [1.0, 1.7, 2.0, 2.4])
def test_library_load_cv_matches_the_oracle(rule, p):
    L = mixed_lengths(7, 3000)
    want = osched.bucket_load_cv(L, synth.BUCKET_S, M_MEM, M_COMP, p, rule)
    got = A.adaln_bucket_load_cv(L, synth.BUCKET_S, M_MEM, M_COMP, p, rule)
    assert got["batches"] == want["batches"]
    assert abs(got["cv"] - want["cv"]) <= 1e-9 * want["cv"]
    assert abs(got["mean"] - want["mean"]) <= 1e-9 * want["mean"]


def test_dual_constraint_caps_the_cost_of_compute_bound_buckets():
    """Where the compute bound binds (S^(p-1) >= M_comp / M_mem: here S >= 4096), an
    equal-token batch costs M_mem * S^(p-1), growing with S, while a dual-constraint batch
    costs at most M_comp (or one sample, S^p, if that alone is above it): on lengths from
    that range the dual rule has the lower maximum cost and the lower imbalance."""
    rng = np.random.default_rng(9)
    L = np.exp(rng.uniform(math.log(2048), math.log(32760), 5000)).astype(np.int64)
    buckets = [4096, 16384, 32760]
    equal = osched.bucket_load_cv(L, buckets, M_MEM, M_COMP, 2.0, 0)
    dual = osched.bucket_load_cv(L, buckets, M_MEM, M_COMP, 2.0, 1)
    assert dual["cv"] < equal["cv"]
    costs = lambda rule: [k * S ** 2 for S, k in osched.batches_of(L, buckets, M_MEM, M_COMP, 2.0, rule)]
    assert max(costs(1)) == max(M_COMP, 32760 ** 2) < max(costs(0))
    for got, want in ((A.adaln_bucket_load_cv(L, buckets, M_MEM, M_COMP, 2.0, r), w)
                      for r, w in ((0, equal), (1, dual))):
        assert abs(got["cv"] - want["cv"]) <= 1e-9 * want["cv"]


def test_load_cv_rejects_bad_arguments():
    with pytest.raises(A.AdalnError):
        A.adaln_bucket_load_cv([5], [2, 4], 8, 16, 2.0, 0)      # longer than every bucket
    with pytest.raises(A.AdalnError):
        A.adaln_bucket_load_cv([1], [4, 2], 8, 16, 2.0, 0)      # buckets not increasing
    with pytest.raises(A.AdalnError):
        A.adaln_bucket_load_cv([1], [2, 4], 8, 16, 2.0, 2)      # no such rule
