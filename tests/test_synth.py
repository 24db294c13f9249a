"""The seeded input generator (shared by both sides): determinism, layout and
the value recipes of the workloads."""
import numpy as np

import synth


def test_normal_is_deterministic_and_counter_based():
    a = synth.normal(7, 3, 1001, 0.0, 1.0, synth.F64)
    b = synth.normal(7, 3, 1001, 0.0, 1.0, synth.F64)
    assert np.array_equal(a, b)
    c = synth.normal(7, 3, 500, 0.0, 1.0, synth.F64)
    assert np.array_equal(a[:500], c)                  # a prefix does not depend on n
    assert not np.array_equal(a, synth.normal(8, 3, 1001, 0.0, 1.0, synth.F64))
    assert not np.array_equal(a, synth.normal(7, 4, 1001, 0.0, 1.0, synth.F64))


def test_normal_moments():
    z = synth.normal(1, 1, 400000, 0.0, 1.0, synth.F64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs(np.mean(z ** 4) - 3) < 0.05             # Gaussian kurtosis
    s = synth.normal(1, 2, 100000, 0.0, 0.02, synth.F64)
    assert abs(s.std() - 0.02) < 0.001


def test_bf16_rounding_matches_oracle(orc):
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e4, 5000),
                        rng.normal(0, 1e-30, 2000), [0.0, -0.0, 3.4e38, -3.4e38, 1e-45]])
    assert np.array_equal(synth.round_bf16(v), orc.round_bf16(v))
    f = synth.normal(5, 1, 1000, 0.0, 1.0, synth.F64)
    assert np.array_equal(synth.normal(5, 1, 1000, 0.0, 1.0, synth.BF16), orc.round_bf16(f))
    assert np.array_equal(synth.normal(5, 1, 1000, 0.0, 1.0, synth.F32), f.astype(np.float32))


def test_scaled_rows_recipe():
    cu = np.array([0, 3000], np.int64)
    x = synth.rows(2, synth.STREAM_X, synth.ROWS_SCALED, cu, 512, synth.F64)
    mu, sd = x.mean(axis=1), x.std(axis=1)
    assert abs(np.std(mu) - 0.5) < 0.05                # offsets ~ N(0, 0.5)
    assert abs(np.std(np.log(sd)) - 0.5) < 0.05        # scales ~ LogNormal(0, 0.5)


def test_adversarial_rows_recipe():
    cu = np.array([0, 40, 100], np.int64)
    x = synth.rows(4, synth.STREAM_X, synth.ROWS_ADVERSARIAL, cu, 64, synth.F32)
    for s in range(2):
        seg = x[cu[s]:cu[s + 1]]
        assert np.all(seg[0] == 0)
        for r in range(1, len(seg)):
            row = seg[r].astype(np.float64)
            if r % 16 == 1:
                assert abs(row.mean()) <= 1000 and row.std() < 0.05
            elif r % 16 == 2:
                assert np.all(row == row[0]) and abs(row[0]) <= 1000
            elif r % 16 == 3:
                if (r // 16) % 2:
                    assert np.all(np.abs(row) == 65504)
                else:
                    assert row.std() > 1e4
    xb = synth.rows(4, synth.STREAM_X, synth.ROWS_ADVERSARIAL, cu, 64, synth.BF16)
    wb = synth.widen(xb, synth.BF16)
    assert wb[3].std() < 100                           # the 65504 class is fp32-only


def test_workload_tables(orc):
    w0 = synth.config(0)
    assert w0.x.shape == (512, 128) and w0.x.dtype == np.float32 and w0.dense == (2, 256)
    w3 = synth.config(3, bucket_batch=__import__("oracle").bucket_batch, generate=False)
    assert w3.nseg == 676 and w3.R == 534344 and w3.meta["batches"] == [512, 128, 32, 2, 1, 1]
    assert np.array_equal(w3.mod_idx, np.arange(676))
    w4 = synth.config(4, generate=False)
    assert w4.cu_seqlens.tolist() == [0, 512, 33272, 33784, 66544]
    assert w4.mod_idx.tolist() == [0, 2, 1, 3] and w4.nmod == 4
