"""Host-side pieces of bench.py that need no GPU: the byte accounting of a step and the
segment chunks of the pipelined end-to-end step."""
import bench
import synth
from oracle import bucket


def test_algorithmic_bytes_per_call():
    R, D, e, nmod = 1000, 3072, 2, 3
    nb = bench.algorithmic_bytes(R, D, e, nmod)
    assert nb["fwd"] == 2 * R * D * e + 8 * R + 2 * nmod * D * e
    assert nb["bwd_partials"] == 3 * R * D * e + 8 * R + nmod * D * e
    assert nb["bwd_reduce"] == 8 * nmod * D
    assert nb["step"] == nb["fwd"] + nb["bwd"]


def test_e2e_chunks_cover_the_packed_batch_in_order():
    w = bench.make_workload("packed", bucket_batch=bucket.bucket_batch, generate=False)
    chunks = bench.e2e_chunks(w, 8)
    assert chunks[0][0] == 0 and chunks[-1][1] == w.nseg
    assert all(a[1] == b[0] for a, b in zip(chunks[:-1], chunks[1:]))
    assert all(s1 > s0 for s0, s1 in chunks)
    tokens = [int(w.cu_seqlens[s1] - w.cu_seqlens[s0]) for s0, s1 in chunks]
    assert sum(tokens) == w.R


def test_e2e_chunks_refuse_shared_or_permuted_tables():
    # Dense batches and tables whose rows are not the segments in order cannot be split
    # into chunks that each own a contiguous, disjoint range of table rows.
    assert bench.e2e_chunks(bench.make_workload("wan-1.3b", generate=False), 8) is None
    assert bench.e2e_chunks(bench.make_workload("mmdit-bf16", generate=False), 8) is None
    w = synth.make("c", 1, synth.BF16, 64, [5, 6, 7], [0, 0, 1], 2, generate=False)
    assert bench.e2e_chunks(w, 2) is None
    # Identity tables split at the first segment boundary at or after each token quantile.
    w = synth.make("c", 1, synth.BF16, 64, [5, 6, 7, 8], None, None, generate=False)
    assert bench.e2e_chunks(w, 2) == [(0, 3), (3, 4)]


def test_literal_bytes_count_each_tensor_once():
    # read x, dy, shift, scale; write y, dx, mean, rstd, dshift, dscale
    R, D, e, nmod = 1000, 3072, 2, 3
    want = (R * D * e) * 4 + 4 * R * 2 + nmod * D * e * 2 + nmod * D * 4 * 2
    assert bench.literal_bytes(R, D, e, nmod) == want
    # Against the per-call sums: x is read by both calls and the statistics are written by
    # the forward and read by the backward, so without modulation rows the calls' row
    # traffic is 5/4 of the literal count's.
    nb = bench.algorithmic_bytes(R, D, e, 0)
    assert nb["step"] - 16 * R == 5 * (bench.literal_bytes(R, D, e, 0) - 8 * R) // 4


def test_oracle_blocks_on_threads_sum_like_one_pass(orc):
    import numpy as np
    w = synth.make("blk", 9, synth.F32, 64, [300, 5, 1200], [1, 0, 1], 2, dy_std=0.5)
    _, mean, rstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod)
    _, dsh, dsc = orc.bwd(w.dy, w.x, mean.astype(np.float32), rstd.astype(np.float32), w.scale, w.dtype,
                          w.cu_seqlens, w.mod_idx, w.nmod)
    bsh, bsc = orc.fwd_bwd_blocks(w.x, w.dy, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod,
                                  (0, w.R), 4, block_rows=100)
    np.testing.assert_allclose(bsh, dsh, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bsc, dsc, rtol=1e-12, atol=1e-12)
