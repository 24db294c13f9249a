"""The dual-constraint bucket size (host integer rule), oracle side.

AdaptiveLoad technical summary, section 2.A: B = max(1, min(floor(M_mem/S),
floor(M_comp/S^p))). The product's C implementation is checked against the
same pins in tests/test_abi.py.
"""
import itertools
import os

import pytest

from oracle.bucket import bucket_batch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bucket_batch_mixed_length.txt")


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(v) for v in line.split()))
    return rows


def brute_force(S, M_mem, M_comp, p):
    """Largest B >= 1 with B*S <= M_mem and B*S^p <= M_comp, by enumeration;
    1 when no B >= 1 satisfies both."""
    best = 0
    B = 1
    while B * S <= M_mem and B * S ** p <= M_comp:
        best = B
        B += 1
    return max(1, best)


def test_golden_table():
    rows = golden_rows()
    assert len(rows) == 6
    for S, M_mem, M_comp, p, B in rows:
        assert bucket_batch(S, M_mem, M_comp, p) == B
    lens = [S for S, _, _, _, B in rows for _ in range(B)]
    assert len(lens) == 676 and sum(lens) == 534344


def test_brute_force_grid():
    for S, M_mem, M_comp, p in itertools.product(range(1, 24), (1, 5, 17, 64, 100),
                                                 (1, 9, 50, 333, 1000), (1, 2, 3)):
        assert bucket_batch(S, M_mem, M_comp, p) == brute_force(S, M_mem, M_comp, p), (S, M_mem, M_comp, p)


def test_edges():
    assert bucket_batch(1, 1, 1, 1) == 1
    assert bucket_batch(10 ** 6, 10, 10, 2) == 1            # S beyond both limits
    assert bucket_batch(2, 2 ** 62, 2 ** 62, 61) == 2        # S^p just at 2^61
    assert bucket_batch(3, 2 ** 62, 2 ** 62, 40) == 1        # S^p beyond 64 bits
    for bad in ((0, 1, 1, 1), (1, 0, 1, 1), (1, 1, 0, 1), (1, 1, 1, 0), (-5, 1, 1, 2)):
        with pytest.raises(ValueError):
            bucket_batch(*bad)
