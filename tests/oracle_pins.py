"""Pins for the CPU oracle: facts that the operator's definition and plain
mathematics fix, checked without retyping the oracle's formulas.

Each pin takes an ``oracle.Oracle`` so the same checks run against the real
oracle (tests/test_oracle_pins.py) and against mutants with a planted mistake
(tests/test_oracle_mutants.py), which must each fail at least one pin.

The operator: AdaptiveLoad technical summary, section 2.B "Fused
LayerNorm-Modulate CUDA kernels" (per-row mean/variance over D, modulation
applied in a third pass; modulation gradients reduced along the sequence).
"""
from __future__ import annotations

import math

import numpy as np

F32, BF16, F64 = 0, 1, 2


def _table(lens):
    cu = np.zeros(len(lens) + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    return cu


def _dense_table(Bt, N):
    return _table([N] * Bt), np.arange(Bt, dtype=np.int64)


def pin_zero_modulation_moments(o):
    """shift = scale = 0: every output row has mean 0 and biased variance
    var/(var + eps), var = numpy's population variance of the input row."""
    rng = np.random.default_rng(11)
    for D, eps in ((64, 1e-6), (96, 0.37), (8, 2.5)):
        x = rng.normal(3.0, 1.7, size=(5, D)) * rng.uniform(0.05, 4.0, size=(5, 1))
        z = np.zeros((1, D))
        cu, mod = _dense_table(1, 5)
        y, mean, rstd = o.fwd(x, z, z, F64, cu, mod, 1, eps=eps)
        v = np.var(x, axis=1)
        assert np.all(np.abs(y.mean(axis=1)) <= 1e-13 * (1 + np.abs(x).max())), "row mean of y != 0"
        np.testing.assert_allclose(np.var(y, axis=1), v / (v + eps), rtol=1e-12, atol=0)
        np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-14, atol=1e-14)


def pin_constant_row(o):
    """A constant row has zero variance: y == shift[m] exactly, mean == c,
    rstd == eps^-1/2."""
    D = 16
    rng = np.random.default_rng(12)
    shift = rng.normal(0, 1, (3, D))
    scale = rng.normal(0, 1, (3, D))
    cs = [0.0, -731.25, 1e3, 3.0]
    x = np.repeat(np.array(cs)[:, None], D, axis=1)
    cu, mod = _table([1, 2, 1]), np.array([2, 0, 1])
    for eps in (1e-6, 0.25):
        y, mean, rstd = o.fwd(x, shift, scale, F64, cu, mod, 3, eps=eps)
        assert np.array_equal(y, shift[[2, 0, 0, 1]]), "constant row must give y == shift"
        assert np.array_equal(mean, np.array(cs))
        np.testing.assert_allclose(rstd, eps ** -0.5, rtol=1e-15)


def pin_d2_closed_form(o):
    """D = 2: x = (a, b) gives xhat = (-h, h) / sqrt(h^2 + eps) with h = (b - a)/2."""
    rng = np.random.default_rng(13)
    x = rng.normal(0, 2, (7, 2))
    x[0] = (5.0, 5.0)
    shift = rng.normal(0, 1, (1, 2))
    scale = rng.normal(0, 1, (1, 2))
    cu, mod = _dense_table(1, 7)
    eps = 0.3
    y, _, _ = o.fwd(x, shift, scale, F64, cu, mod, 1, eps=eps)
    h = (x[:, 1] - x[:, 0]) / 2
    xh = np.stack([-h, h], axis=1) / np.sqrt(h * h + eps)[:, None]
    np.testing.assert_allclose(y, xh * (1 + scale) + shift, rtol=1e-13, atol=1e-14)


def pin_translation_invariance(o):
    """x -> x + c leaves y unchanged (up to the rounding of x + c itself)."""
    rng = np.random.default_rng(14)
    D = 48
    x = rng.normal(0, 1, (4, D))
    shift, scale = rng.normal(0, 1, (1, D)), rng.normal(0, 1, (1, D))
    cu, mod = _dense_table(1, 4)
    y0, m0, r0 = o.fwd(x, shift, scale, F64, cu, mod, 1)
    for c in (7.0, -250.0, 1e4):
        y1, m1, r1 = o.fwd(x + c, shift, scale, F64, cu, mod, 1)
        np.testing.assert_allclose(y1, y0, rtol=0, atol=1e-10 * (1 + abs(c)))
        np.testing.assert_allclose(r1, r0, rtol=1e-10 * (1 + abs(c)))
        np.testing.assert_allclose(m1, m0 + c, rtol=1e-14)


def pin_scale_invariance(o):
    """x -> a*x with eps -> a^2*eps gives xhat -> sign(a)*xhat exactly (with eps
    fixed the factor is sqrt((var+eps)/(var+eps/a^2)), checked too)."""
    rng = np.random.default_rng(15)
    D = 40
    x = rng.normal(1, 1, (3, D))
    z = np.zeros((1, D))
    cu, mod = _dense_table(1, 3)
    eps = 0.05
    y0, _, _ = o.fwd(x, z, z, F64, cu, mod, 1, eps=eps)
    v = np.var(x, axis=1)
    for a in (3.0, -2.0, 1e-3):
        y1, _, _ = o.fwd(a * x, z, z, F64, cu, mod, 1, eps=eps * a * a)
        np.testing.assert_allclose(y1, np.sign(a) * y0, rtol=1e-11, atol=1e-13)
        y2, _, _ = o.fwd(a * x, z, z, F64, cu, mod, 1, eps=eps)
        f = np.sqrt((v + eps) / (v + eps / (a * a)))
        np.testing.assert_allclose(y2, np.sign(a) * y0 * f[:, None], rtol=1e-11, atol=1e-13)


def pin_modulation_is_affine(o):
    """For a token of modulation row m, (y - shift[m]) / (1 + scale[m]) is the
    normalised row: mean 0, variance var/(var+eps). Segments pick their row through
    mod_idx (a permutation here, with one row used twice and one row unused)."""
    rng = np.random.default_rng(16)
    D, eps = 32, 0.2
    lens = [3, 1, 4, 2]
    mod = np.array([3, 0, 3, 1])
    cu = _table(lens)
    x = rng.normal(0, 1, (cu[-1], D)) * 2 + 1
    shift = rng.normal(0, 1, (5, D))
    scale = rng.normal(0, 0.5, (5, D))
    y, _, _ = o.fwd(x, shift, scale, F64, cu, mod, 5, eps=eps)
    m_of_row = np.repeat(mod, lens)
    xh = (y - shift[m_of_row]) / (1 + scale[m_of_row])
    v = np.var(x, axis=1)
    assert np.all(np.abs(xh.mean(axis=1)) < 1e-12)
    np.testing.assert_allclose(np.var(xh, axis=1), v / (v + eps), rtol=1e-11)


def pin_packed_equals_per_segment(o):
    """A packed call over several segments equals one call per segment with a
    one-row modulation table (the trivial mapping)."""
    rng = np.random.default_rng(17)
    D = 24
    lens = [2, 0, 5, 1, 3]
    mod = np.array([2, 1, 0, 2, 1])
    cu = _table(lens)
    x = rng.normal(0, 1, (cu[-1], D))
    dy = rng.normal(0, 1, (cu[-1], D))
    shift, scale = rng.normal(0, 1, (3, D)), rng.normal(0, 1, (3, D))
    y, mean, rstd = o.fwd(x, shift, scale, F64, cu, mod, 3)
    dx, dsh, dsc = o.bwd(dy, x, mean, rstd, scale, F64, cu, mod, 3)
    dsh_ref, dsc_ref = np.zeros((3, D)), np.zeros((3, D))
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        m = mod[s]
        one = (np.array([0, L]), np.array([0]))
        ys, ms, rs = o.fwd(x[a:b], shift[m:m + 1], scale[m:m + 1], F64, *one, 1)
        assert np.array_equal(ys, y[a:b]) and np.array_equal(ms, mean[a:b])
        dxs, dshs, dscs = o.bwd(dy[a:b], x[a:b], ms, rs, scale[m:m + 1], F64, *one, 1)
        assert np.array_equal(dxs, dx[a:b])
        dsh_ref[m] += dshs[0]
        dsc_ref[m] += dscs[0]
    np.testing.assert_allclose(dsh, dsh_ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dsc, dsc_ref, rtol=1e-14, atol=1e-14)


def _loss(o, x, shift, scale, dy, cu, mod, nmod, eps):
    y, _, _ = o.fwd(x, shift, scale, F64, cu, mod, nmod, eps=eps)
    return math.fsum((dy * y).ravel())


def pin_finite_differences(o):
    """Backward == central finite differences of L = sum(dy * y) in double,
    w.r.t. x, shift and scale, on a tiny packed problem (2 segments, D = 8)."""
    rng = np.random.default_rng(18)
    D = 8
    lens, mod, nmod = [3, 2], np.array([1, 0]), 2
    cu = _table(lens)
    R = int(cu[-1])
    x = rng.normal(0.5, 1.3, (R, D))
    dy = rng.normal(0, 1, (R, D))
    shift, scale = rng.normal(0, 0.5, (nmod, D)), rng.normal(0, 0.5, (nmod, D))
    for eps in (1e-6, 0.3):
        _, mean, rstd = o.fwd(x, shift, scale, F64, cu, mod, nmod, eps=eps)
        dx, dsh, dsc = o.bwd(dy, x, mean, rstd, scale, F64, cu, mod, nmod)

        def num(arr, setter):
            g = np.zeros_like(arr)
            for idx in np.ndindex(*arr.shape):
                h = 1e-6 * max(1.0, abs(arr[idx]))
                a = arr.copy(); a[idx] += h
                b = arr.copy(); b[idx] -= h
                g[idx] = (setter(a) - setter(b)) / (2 * h)
            return g

        gx = num(x, lambda a: _loss(o, a, shift, scale, dy, cu, mod, nmod, eps))
        gsh = num(shift, lambda a: _loss(o, x, a, scale, dy, cu, mod, nmod, eps))
        gsc = num(scale, lambda a: _loss(o, x, shift, a, dy, cu, mod, nmod, eps))
        np.testing.assert_allclose(dx, gx, rtol=2e-6, atol=2e-7)
        np.testing.assert_allclose(dsh, gsh, rtol=2e-6, atol=2e-7)
        np.testing.assert_allclose(dsc, gsc, rtol=2e-6, atol=2e-7)


def pin_dx_identities(o):
    """sum_d dx = 0 exactly (in exact arithmetic), and
    sum_d dx * xhat = D * rstd * mean(g*xhat) * eps / (var + eps)."""
    rng = np.random.default_rng(19)
    D = 64
    x = rng.normal(2, 1.5, (6, D))
    dy = rng.normal(0, 1, (6, D))
    shift, scale = rng.normal(0, 1, (1, D)), rng.normal(0, 0.3, (1, D))
    cu, mod = _dense_table(1, 6)
    for eps in (1e-6, 0.9):
        _, mean, rstd = o.fwd(x, shift, scale, F64, cu, mod, 1, eps=eps)
        dx, _, _ = o.bwd(dy, x, mean, rstd, scale, F64, cu, mod, 1)
        assert np.all(np.abs(dx.sum(axis=1)) <= 1e-12 * np.abs(dx).sum(axis=1))
        xh = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(np.var(x, axis=1, keepdims=True) + eps)
        g = dy * (1 + scale)
        v = np.var(x, axis=1)
        want = D * rstd * (g * xh).mean(axis=1) * eps / (v + eps)
        np.testing.assert_allclose((dx * xh).sum(axis=1), want, rtol=1e-8, atol=1e-12)


def pin_dshift_is_exact_column_sum(o):
    """dshift[m, d] == the exact (error-free) sum of dy[:, d] over m's tokens.
    dy values are multiples of 2^-8 below 2^10, so every partial sum is exact in
    double and the comparison is bitwise."""
    rng = np.random.default_rng(20)
    D = 12
    lens, mod, nmod = [40, 7, 13, 0], np.array([1, 0, 1, 2]), 3
    cu = _table(lens)
    R = int(cu[-1])
    dy = rng.integers(-2 ** 17, 2 ** 17, (R, D)).astype(np.float64) / 256.0
    x = rng.normal(0, 1, (R, D))
    scale = rng.normal(0, 1, (nmod, D))
    _, mean, rstd = o.fwd(x, scale, scale, F64, cu, mod, nmod)
    _, dsh, _ = o.bwd(dy, x, mean, rstd, scale, F64, cu, mod, nmod)
    m_of_row = np.repeat(mod, lens)
    for m in range(nmod):
        for d in range(D):
            assert dsh[m, d] == math.fsum(dy[m_of_row == m, d])


def pin_storage_dtypes_widen_exactly(o):
    """bf16 and fp32 inputs are read as their exact values: the same values given
    as float64 give identical outputs."""
    rng = np.random.default_rng(21)
    D = 16
    vals = rng.normal(0, 3, (4, D)).astype(np.float32)
    bf_bits = (vals.view(np.uint32) >> 16).astype(np.uint16)   # truncation: exact bf16 values
    bf_vals = (bf_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    cu, mod = _dense_table(2, 2)
    sh = rng.normal(0, 1, (2, D)).astype(np.float32)
    sh_bits = (sh.view(np.uint32) >> 16).astype(np.uint16)
    sh_vals = (sh_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = o.fwd(bf_bits, sh_bits, sh_bits, BF16, cu, mod, 2)
    b = o.fwd(bf_vals, sh_vals, sh_vals, F64, cu, mod, 2)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    a = o.fwd(vals, sh, sh, F32, cu, mod, 2)
    b = o.fwd(vals.astype(np.float64), sh.astype(np.float64), sh.astype(np.float64), F64, cu, mod, 2)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    dy = rng.normal(0, 1, (4, D)).astype(np.float32)
    dy_bits = (dy.view(np.uint32) >> 16).astype(np.uint16)
    dy_vals = (dy_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    _, mean, rstd = b
    a = o.bwd(dy_bits, bf_bits, mean, rstd, sh_bits, BF16, cu, mod, 2)
    b = o.bwd(dy_vals, bf_vals, mean, rstd, sh_vals, F64, cu, mod, 2)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def _all_finite_bf16():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), vals


def pin_round_bf16(o):
    """double -> bf16 is round-to-nearest-even, in one step:
    every bf16 value maps to itself; a midpoint between neighbours goes to the one
    with an even last bit; anything strictly off a midpoint goes to the nearer
    neighbour; the top of the range overflows to infinity; signs are kept."""
    bits, vals = _all_finite_bf16()
    assert np.array_equal(o.round_bf16(vals), bits)
    assert np.array_equal(o.round_bf16(-vals), bits | 0x8000)
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2                                   # exact in double
    even = np.where(bits[:-1] % 2 == 0, bits[:-1], bits[1:])
    assert np.array_equal(o.round_bf16(mid), even)
    gap = hi - lo
    assert np.array_equal(o.round_bf16(mid - gap / 1024), bits[:-1])
    assert np.array_equal(o.round_bf16(mid + gap / 1024), bits[1:])
    top = vals[-1]
    ulp_top = top - vals[-2]
    assert o.round_bf16([top + ulp_top / 2])[0] == 0x7F80          # tie rounds to even = inf
    assert o.round_bf16([top + ulp_top / 2 - ulp_top / 64])[0] == 0x7F7F
    assert o.round_bf16([float("inf"), -float("inf")]).tolist() == [0x7F80, 0xFF80]
    assert o.round_bf16([2.0 ** -134])[0] == 0x0000                # half the smallest subnormal: tie to 0
    assert o.round_bf16([2.0 ** -134 * 1.0000001])[0] == 0x0001
    assert o.round_bf16([-0.0])[0] == 0x8000
    # a value one fp32 ulp above a bf16 midpoint: double rounding through fp32 would tie
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert o.round_bf16([x])[0] == 0x3F81


ALL_PINS = [
    pin_zero_modulation_moments,
    pin_constant_row,
    pin_d2_closed_form,
    pin_translation_invariance,
    pin_scale_invariance,
    pin_modulation_is_affine,
    pin_packed_equals_per_segment,
    pin_finite_differences,
    pin_dx_identities,
    pin_dshift_is_exact_column_sum,
    pin_storage_dtypes_widen_exactly,
    pin_round_bf16,
]
