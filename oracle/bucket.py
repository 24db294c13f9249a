"""TEST INFRASTRUCTURE ONLY: the dual-constraint bucket size, as a plain definition.

AdaptiveLoad technical summary, section 2.A "Dual-constraint adaptive load
balancing": a bucket of sequence length S holds B sequences, limited at once by
memory (B * S <= M_mem) and by compute (B * S^p <= M_comp, p the fitted exponent
of the step-time model), and never fewer than one:

    B = max(1, min(floor(M_mem / S), floor(M_comp / S^p)))

Python integers are unbounded, so S**p and both floors are exact.
"""


def bucket_batch(S: int, M_mem: int, M_comp: int, p: int) -> int:
    if S <= 0 or M_mem <= 0 or M_comp <= 0 or p < 1:
        raise ValueError("bucket_batch needs S, M_mem, M_comp > 0 and p >= 1")
    return max(1, min(M_mem // S, M_comp // S ** p))
