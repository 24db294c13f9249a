"""CUDA path (through the C-ABI binding) against the CPU oracle on the same seeded bits.

Every case is compared element by element on every row: small problems (several row
tiles, ragged tails, odd segment tables, every row-width code path and staging mode) and
the full-size workloads in the launch configuration the benchmark uses, including each
bucket of the packed workload as its own call. The oracle runs a chunk of rows at a time
on a thread pool.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaln_layernorm_modulate_gb300 as A
    A.lib()  # loads the in-tree libadaln.so or raises


def _run_and_compare(orc, w):
    """Forward, then two backwards: one on the oracle's statistics rounded to fp32 (isolated,
    strict tolerance) and one on the GPU forward's own statistics (pipeline, plus the bound of
    a one-ulp mean shift). Every row of y, mean, rstd and dx and every row of dshift/dscale
    is compared with the oracle."""
    t = H.torch()
    d = H.upload(w)
    y, mean, rstd, st = H.gpu_fwd(d)
    assert st == 0
    dx2, dsh2, dsc2, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    y_h, mean_h, rstd_h = H.to_host(y, w.dtype), H.to_host(mean, 0), H.to_host(rstd, 0)
    pipeline = (H.to_host(dx2, w.dtype), H.to_host(dsh2, 0), H.to_host(dsc2, 0))
    del y, dx2
    m32, r32 = H.forward_all_rows(orc, w, y_h, mean_h, rstd_h)
    del y_h
    dm = t.from_numpy(m32.astype(np.float32)).cuda()
    dr = t.from_numpy(r32.astype(np.float32)).cuda()
    dx, dsh, dsc, st = H.gpu_bwd(d, dm, dr)
    assert st == 0
    isolated = (H.to_host(dx, w.dtype), H.to_host(dsh, 0), H.to_host(dsc, 0))
    del d, dx
    t.cuda.empty_cache()
    H.backward_all_rows(orc, w, m32, r32, pipeline=pipeline, isolated=isolated)


SMALL = {
    "tiny-f32-2x256x128": lambda: synth.config(0),
    "dense-bf16-2x300x1536": lambda: synth.dense("c", 101, synth.BF16, 2, 300, 1536,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "dense-bf16-1x333x5120": lambda: synth.dense("c", 102, synth.BF16, 1, 333, 5120,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "dense-f32-2x129x3072": lambda: synth.dense("c", 103, synth.F32, 2, 129, 3072,
                                                x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-bf16-d3072-ragged": lambda: synth.make("c", 104, synth.BF16, 3072,
                                                   [1, 7, 256, 1000, 3, 0, 513],
                                                   [4, 0, 2, 2, 5, 1, 0], 6,
                                                   x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-f32-d3072-adversarial": lambda: synth.make("c", 105, synth.F32, 3072, [40, 300, 17, 129],
                                                       [0, 2, 1, 3], 4, x_mode=synth.ROWS_ADVERSARIAL,
                                                       mod_std=0.5, dy_std=0.02),
    "packed-bf16-d3072-adversarial": lambda: synth.make("c", 106, synth.BF16, 3072, [40, 300, 17, 129],
                                                        [0, 2, 1, 3], 4, x_mode=synth.ROWS_ADVERSARIAL,
                                                        mod_std=0.5, dy_std=0.02),
    "dense-bf16-d8": lambda: synth.dense("c", 107, synth.BF16, 3, 50, 8),
    "dense-bf16-2x200x768": lambda: synth.dense("c", 118, synth.BF16, 2, 200, 768,
                                                x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-bf16-d264": lambda: synth.make("c", 108, synth.BF16, 264, [5, 90, 33], [1, 1, 0], 2),
    "dense-bf16-d16384": lambda: synth.dense("c", 109, synth.BF16, 1, 40, 16384, dy_std=0.1),
    "dense-f32-d8192": lambda: synth.dense("c", 110, synth.F32, 1, 33, 8192),
    # A backward ring of two rounds over the 150 KB budget (2 x 96 KB): fp32 D=12288.
    "dense-f32-2x17x12288": lambda: synth.dense("c", 121, synth.F32, 2, 17, 12288, dy_std=0.1),
    # bf16 rows of 8 vectors a thread over 7 warps (D=14336) and of 10240 (an exact cover
    # away from the forward's preferred 6 vectors a thread).
    "dense-bf16-1x37x14336": lambda: synth.dense("c", 122, synth.BF16, 1, 37, 14336, dy_std=0.1),
    "packed-bf16-d10240": lambda: synth.make("c", 123, synth.BF16, 10240, [20, 1, 25], [0, 1, 0], 2,
                                             x_mode=synth.ROWS_SCALED, dy_std=0.02),
    # fp32 D=14336: a two-round backward ring of 224 KB, near the per-CTA shared-memory limit.
    "dense-f32-2x19x14336": lambda: synth.dense("c", 124, synth.F32, 2, 19, 14336, dy_std=0.1),
    # fp32 rows too wide for a two-round backward ring: the split form (two-CTA clusters,
    # half a row each, row sums exchanged through distributed shared memory); a few rows, many
    # rows a tile (the exchange buffers cycle), and a packed table of a width the threads do
    # not cover exactly (D=15360: 240 of 256 lanes) with shared modulation rows.
    "dense-f32-2x21x16384": lambda: synth.dense("c", 119, synth.F32, 2, 21, 16384, dy_std=0.1),
    "dense-f32-1x1500x16384-split": lambda: synth.dense("c", 127, synth.F32, 1, 1500, 16384,
                                                        x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-f32-d15360-split": lambda: synth.make("c", 128, synth.F32, 15360, [700, 3, 0, 250, 47],
                                                  [1, 0, 2, 1, 1], 3, x_mode=synth.ROWS_SCALED,
                                                  dy_std=0.02),
    # The narrowest split width: fp32 D=14344, half a row = 1793 vectors over 256 threads
    # (thread t owns vectors t + 256k: eight for thread 0, seven for the others).
    "packed-f32-d14344-split-narrowest": lambda: synth.make("c", 129, synth.F32, 14344, [300, 1, 77],
                                                            [0, 1, 0], 2, x_mode=synth.ROWS_SCALED,
                                                            dy_std=0.02),
    "packed-f32-d128-many": lambda: synth.make(
        "c", 111, synth.F32, 128, list(np.random.default_rng(5).integers(0, 10, 100)),
        list(np.random.default_rng(6).integers(0, 13, 100)), 13),
    "dense-f32-one-row": lambda: synth.dense("c", 112, synth.F32, 1, 1, 1536),
    # Many short samples: few pieces per modulation row, so row-major partials and the
    # row-major stage 2 of a dense batch.
    "dense-bf16-800x5x1024": lambda: synth.dense("c", 125, synth.BF16, 800, 5, 1024,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    # The backward's wide form (bf16 D=16384, 4 x 512 threads) on a packed table whose
    # modulation rows are shared and whose segments end inside tiles.
    "packed-bf16-d16384-wide": lambda: synth.make("c", 126, synth.BF16, 16384, [30, 2, 9, 0, 41],
                                                  [1, 0, 1, 2, 0], 3, x_mode=synth.ROWS_SCALED,
                                                  dy_std=0.02),
    # More segments than stage 2 examines in one pass of the table (1024), rows of the
    # modulation table whose segments fall in several passes, and empty segments.
    "packed-f32-d64-3000seg": lambda: synth.make(
        "c", 113, synth.F32, 64, list(np.random.default_rng(7).integers(0, 10, 3000)),
        list(np.random.default_rng(8).integers(0, 40, 3000)), 41),
    # Tiles of hundreds of thousands of narrow rows: many rounds of the forward's bulk ring.
    "packed-bf16-d8-long-tiles": lambda: synth.make(
        "c", 115, synth.BF16, 8, [400000, 3, 700000], [1, 0, 1], 2,
        x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "dense-f32-d16-long-tiles": lambda: synth.dense("c", 116, synth.F32, 2, 600000, 16),
    # Many modulation rows over a 700-segment table: rows shared by several segments, rows
    # no segment uses (zero gradients), stage 2 over 2 column blocks x 601 rows.
    "packed-f32-d2048-601rows": lambda: synth.make(
        "c", 117, synth.F32, 2048, list(np.random.default_rng(12).integers(0, 30, 700)),
        list(np.random.default_rng(13).integers(0, 601, 700)), 601, dy_std=0.5),
    # One long segment spread over many row tiles, sharing its modulation row with
    # thousands of short ones.
    # 90,008 bf16 rows of D=3072: more than 64 rows a resident CTA slot on GB300 (912 slots),
    # so the forward stages them with its per-thread copy ring and maps them 3 x 128 threads,
    # as on the packed benchmark workload; rows of two segments share modulation rows.
    "packed-bf16-d3072-copy-ring": lambda: synth.make(
        "c", 120, synth.BF16, 3072, [40000, 7, 50000, 1], [0, 1, 0, 1], 2,
        x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-bf16-d256-long-and-many": lambda: synth.make(
        "c", 114, synth.BF16, 256, [5000] + list(np.random.default_rng(9).integers(1, 8, 2500)),
        [0] + list(np.random.default_rng(10).integers(0, 3, 2500)), 3,
        x_mode=synth.ROWS_SCALED, dy_std=0.02),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_elementwise(orc, name):
    _run_and_compare(orc, SMALL[name]())


def _full_size(orc, w):
    _run_and_compare(orc, w)
    H.torch().cuda.empty_cache()


def test_full_wan_1_3b(orc):
    _full_size(orc, synth.config(1))


def test_full_wan_14b(orc):
    _full_size(orc, synth.config(2))


def test_full_packed_buckets(orc):
    import adaln_layernorm_modulate_gb300 as A
    w = synth.config(3, bucket_batch=A.adaln_bucket_batch)
    assert w.meta["batches"] == [512, 128, 32, 2, 1, 1]
    _full_size(orc, w)


@pytest.mark.parametrize("S", synth.BUCKET_S)
def test_full_bucket_alone(orc, S):
    # Each bucket of the packed workload as its own packed call: bucket_batch(S) segments of
    # S tokens (S = 32760 and 75600: one segment spanning every row tile).
    import adaln_layernorm_modulate_gb300 as A
    w = synth.bucket(S, A.adaln_bucket_batch)
    assert w.nseg == A.adaln_bucket_batch(S, synth.BUCKET_M_MEM, synth.BUCKET_M_COMP, synth.BUCKET_P)
    _full_size(orc, w)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16], ids=["f32", "bf16"])
def test_full_mmdit(orc, dtype):
    _full_size(orc, synth.config(4, dtype=dtype))


def test_shuffled_segment_order_gives_the_same_rows(orc):
    """The packed workload with its 676 segments in a seeded random order (each segment
    keeping its rows and its modulation row) gives, per segment, bitwise the y, mean, rstd
    and dx of the ascending-order call: the row count and so the tiles' length and row
    mapping are the same, and a row's arithmetic does not depend on which tile holds it.
    dshift/dscale sum over other tile pieces, so they are compared with the oracle's."""
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = synth.config(3, bucket_batch=A.adaln_bucket_batch)
    perm = np.random.default_rng(2024).permutation(w.nseg)
    lens = np.diff(w.cu_seqlens)
    cu_p = np.zeros(w.nseg + 1, dtype=np.int64)
    cu_p[1:] = np.cumsum(lens[perm])
    # Row i of the shuffled batch is row src[i] of the ascending one.
    src = np.concatenate([np.arange(w.cu_seqlens[s], w.cu_seqlens[s + 1]) for s in perm])
    d = H.upload(w)
    y, mean, rstd, st = H.gpu_fwd(d)
    assert st == 0
    dx, dsh, dsc, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    idx = t.from_numpy(src).cuda()
    ws = synth.Workload("shuffled", w.seed, w.dtype, w.D, cu_p, w.mod_idx[perm].copy(), w.nmod,
                        x=None, dy=None, shift=w.shift, scale=w.scale)
    dp = H.DevWorkload(ws, d.x[idx], d.dy[idx], d.shift, d.scale,
                       t.from_numpy(cu_p.astype(np.int32)).cuda(),
                       t.from_numpy(ws.mod_idx.astype(np.int32)).cuda())
    y2, mean2, rstd2, st = H.gpu_fwd(dp)
    assert st == 0
    assert t.equal(y2, y[idx]) and t.equal(mean2, mean[idx]) and t.equal(rstd2, rstd[idx])
    del y, y2, d.x
    t.cuda.empty_cache()
    dx2, dsh2, dsc2, st = H.gpu_bwd(dp, mean2, rstd2)
    assert st == 0
    assert t.equal(dx2, dx[idx])
    del dx, dx2, dp, d
    t.cuda.empty_cache()
    # The gradients of every modulation row against the oracle on the ascending rows (the
    # same token sets), with the GPU forward's statistics in both orders being bitwise equal.
    m32, r32 = H.round_f32(H.to_host(mean, 0).astype(np.float64)), H.round_f32(H.to_host(rstd, 0).astype(np.float64))
    ref_sh, ref_sc = H.backward_all_rows(orc, w, m32, r32)
    for got, ref in ((dsh2, ref_sh), (dsc2, ref_sc)):
        g = H.to_host(got, 0)
        for m in range(w.nmod):
            assert H.rel_l2(g[m], ref[m]) <= H.grad_tol(w.dtype), m


def test_backward_is_bitwise_deterministic():
    for w in (synth.dense("det", 201, synth.BF16, 1, 4000, 1536, x_mode=synth.ROWS_SCALED, dy_std=0.02),
              synth.make("det", 202, synth.BF16, 3072, [300, 5, 2000, 77], [1, 0, 1, 2], 3,
                         x_mode=synth.ROWS_SCALED, dy_std=0.02),
              synth.make("det", 203, synth.F32, 16384, [400, 9, 600], [0, 1, 0], 2,
                         x_mode=synth.ROWS_SCALED, dy_std=0.02)):
        d = H.upload(w)
        y, mean, rstd, _ = H.gpu_fwd(d)
        ref = [H.to_host(v, w.dtype if i == 0 else 0) for i, v in enumerate(H.gpu_bwd(d, mean, rstd)[:3])]
        for _ in range(4):
            y2, mean2, rstd2, _ = H.gpu_fwd(d)
            assert H.torch().equal(y, y2) and H.torch().equal(mean, mean2)
            got = [H.to_host(v, w.dtype if i == 0 else 0) for i, v in enumerate(H.gpu_bwd(d, mean, rstd)[:3])]
            for a, b in zip(ref, got):
                assert np.array_equal(a, b)


def test_packed_equals_dense_streams():
    """The MMDiT packed call (4 segments) gives bitwise the per-row results of the dense
    per-stream calls: row math does not depend on which tile holds the row."""
    t = H.torch()
    T, V, D = 64, 700, 3072
    w = synth.make("mm", 301, synth.BF16, D, [T, V, T, V], [0, 2, 1, 3], 4,
                   x_mode=synth.ROWS_ADVERSARIAL, mod_std=0.5, dy_std=0.02)
    d = H.upload(w)
    y, mean, rstd, st = H.gpu_fwd(d)
    dx, dsh, dsc, _ = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    cu = w.cu_seqlens
    for rows_of, table_rows, N in (([0, 2], [0, 1], T), ([1, 3], [2, 3], V)):
        xs = np.concatenate([w.x[cu[s]:cu[s + 1]] for s in rows_of])
        dys = np.concatenate([w.dy[cu[s]:cu[s + 1]] for s in rows_of])
        ws = synth.Workload("stream", 0, w.dtype, D, np.array([0, N, 2 * N]), np.array([0, 1]), 2,
                            dense=(2, N), x=xs, dy=dys, shift=w.shift[table_rows], scale=w.scale[table_rows])
        dd = H.upload(ws)
        y2, mean2, rstd2, _ = H.gpu_fwd(dd)
        dx2, dsh2, dsc2, _ = H.gpu_bwd(dd, mean2, rstd2)
        idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in rows_of])
        it = t.from_numpy(idx).cuda()
        assert t.equal(y[it], y2) and t.equal(mean[it], mean2) and t.equal(rstd[it], rstd2)
        assert t.equal(dx[it], dx2)
        np.testing.assert_allclose(H.to_host(dsh[table_rows], 0), H.to_host(dsh2, 0), rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(H.to_host(dsc[table_rows], 0), H.to_host(dsc2, 0), rtol=1e-5, atol=1e-5)


def test_malformed_tables_report_status_without_faulting():
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = synth.make("bad", 401, synth.BF16, 256, [10, 20, 30], [0, 1, 2], 3)
    d = H.upload(w)
    good_cu, good_mod = d.cu.clone(), d.mod.clone()
    cases = [
        ("decreasing", lambda: d.cu.copy_(t.tensor([0, 25, 5, 60], dtype=t.int32)), A.STATUS[6]),
        ("short total", lambda: d.cu.copy_(t.tensor([0, 10, 30, 50], dtype=t.int32)), A.STATUS[6]),
        ("nonzero start", lambda: d.cu.copy_(t.tensor([3, 10, 30, 60], dtype=t.int32)), A.STATUS[6]),
        ("beyond total", lambda: d.cu.copy_(t.tensor([0, 10, 90, 60], dtype=t.int32)), A.STATUS[6]),
        ("mod too large", lambda: d.mod.copy_(t.tensor([0, 3, 2], dtype=t.int32)), A.STATUS[7]),
        ("mod negative", lambda: d.mod.copy_(t.tensor([-1, 1, 2], dtype=t.int32)), A.STATUS[7]),
    ]
    for name, corrupt, want in cases:
        d.cu.copy_(good_cu)
        d.mod.copy_(good_mod)
        corrupt()
        _, mean, rstd, st = H.gpu_fwd(d)
        assert A.STATUS[st] == want, (name, A.STATUS[st])
        _, _, _, st = H.gpu_bwd(d, mean, rstd)
        assert A.STATUS[st] == want, (name, A.STATUS[st])
        t.cuda.synchronize()
    d.cu.copy_(good_cu)
    d.mod.copy_(good_mod)
    _, mean, rstd, st = H.gpu_fwd(d)
    assert st == 0
    assert H.gpu_bwd(d, mean, rstd)[3] == 0


def test_status_words_decode_with_precedence():
    """adaln_read_status on workspace words written from the host: the per-CTA bits a
    kernel can record (1 cu_seqlens, 2 mod_idx, 4 copy timeout) map to their status, the
    table errors first; a header without the magic reads as a missing status."""
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()

    def status(words, magic=0x4E4C4441):
        head = np.zeros(64, dtype=np.uint32)  # 256-byte header: magic, word count, padding
        head[0], head[1] = magic, len(words)
        buf = np.concatenate([head, np.asarray(words, dtype=np.uint32)])
        ws = t.from_numpy(buf.view(np.uint8)).cuda()
        return A.STATUS[A.adaln_read_status(ws)]

    assert status([0, 0, 0]) == "ADALN_OK"
    assert status([0, 4, 0]) == "ADALN_ERR_TIMEOUT"
    assert status([4, 2, 0]) == "ADALN_ERR_BAD_MOD_IDX"
    assert status([4, 2, 1]) == "ADALN_ERR_BAD_SEQLENS"
    assert status([0, 4], magic=0) == "ADALN_ERR_WORKSPACE"
    assert status([]) == "ADALN_ERR_WORKSPACE"


def test_empty_and_zero_length_segments(orc):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    # Dense backward over no tokens: zero gradients.
    D = 512
    dsh = t.full((3, D), 7.0, device="cuda")
    dsc = t.full((3, D), 7.0, device="cuda")
    nb = A.adaln_bwd_workspace_size(3, 0, D, A.ADALN_BF16)
    ws = t.empty(nb, dtype=t.uint8, device="cuda")
    A.adaln_bwd(None, None, None, None, None, None, dsh, dsc, ws, nb, 3, 0, D, A.ADALN_BF16)
    assert t.count_nonzero(dsh) == 0 and t.count_nonzero(dsc) == 0
    # Packed tables whose segments are all empty.
    w = synth.make("empty", 501, synth.F32, D, [0, 0, 0], [0, 1, 1], 2)
    d = H.upload(w)
    _, mean, rstd, st = H.gpu_fwd(d)
    assert st == 0
    _, dsh, dsc, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0 and t.count_nonzero(dsh) == 0 and t.count_nonzero(dsc) == 0
    # Empty segments between non-empty ones, leading and trailing.
    _run_and_compare(orc, synth.make("gaps", 502, synth.F32, D, [0, 3, 0, 0, 5, 0], [0, 1, 2, 0, 1, 2], 3))


def test_outputs_stay_inside_their_buffers():
    """Guard bands around every output keep their fill pattern."""
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = synth.make("guard", 601, synth.BF16, 1536, [3, 130, 1, 66], [2, 0, 1, 1], 3,
                   x_mode=synth.ROWS_SCALED, dy_std=0.02)
    d = H.upload(w)
    G = 4096  # guard elements on each side (multiple of 8 keeps 16-byte alignment)

    def guarded(n, dtype):
        buf = t.empty(n + 2 * G, dtype=dtype, device="cuda")
        buf.view(t.uint8).fill_(0xA5) if dtype != t.float32 else buf.view(t.int32).fill_(0x5A5A5A5A)
        return buf, buf[G:G + n]

    def intact(buf, n):
        raw = buf.view(t.uint8) if buf.dtype != t.float32 else buf.view(t.int32)
        k = raw.numel() // buf.numel()
        head, tail = raw[:G * k], raw[(G + n) * k:]
        want = 0xA5 if buf.dtype != t.float32 else 0x5A5A5A5A
        return bool((head == want).all()) and bool((tail == want).all())

    yb, y = guarded(w.R * w.D, t.bfloat16)
    mb, mean = guarded(w.R, t.float32)
    rb, rstd = guarded(w.R, t.float32)
    nb = A.adaln_fwd_varlen_workspace_size(w.R, w.nseg, w.D, w.dtype)
    ws = t.empty(nb, dtype=t.uint8, device="cuda")
    A.adaln_fwd_varlen(d.x, d.shift, d.scale, y, mean, rstd, d.cu, d.mod, w.nseg, w.R, w.nmod, w.D,
                       H.EPS, ws, nb, w.dtype)
    dxb, dx = guarded(w.R * w.D, t.bfloat16)
    shb, dsh = guarded(w.nmod * w.D, t.float32)
    scb, dsc = guarded(w.nmod * w.D, t.float32)
    nb = A.adaln_bwd_varlen_workspace_size(w.R, w.nseg, w.nmod, w.D, w.dtype)
    ws2 = t.empty(nb, dtype=t.uint8, device="cuda")
    A.adaln_bwd_varlen(d.dy, d.x, mean, rstd, d.scale, dx, dsh, dsc, d.cu, d.mod, w.nseg, w.R, w.nmod,
                       w.D, ws2, nb, w.dtype)
    t.cuda.synchronize()
    for buf, n in ((yb, w.R * w.D), (mb, w.R), (rb, w.R), (dxb, w.R * w.D), (shb, w.nmod * w.D),
                   (scb, w.nmod * w.D)):
        assert intact(buf, n)


@pytest.mark.parametrize("name", ["dense-bf16-2x300x1536", "packed-bf16-d3072-ragged",
                                  "packed-f32-d3072-adversarial", "dense-bf16-d16384",
                                  "packed-bf16-d8-long-tiles", "packed-bf16-d3072-copy-ring",
                                  "packed-f32-d15360-split"])
def test_recomputed_statistics_are_bitwise_the_saved_ones(name):
    """A backward that recomputes mean/rstd from x gives bitwise the dx, dshift and dscale of
    the backward that reads the forward's saved statistics."""
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = SMALL[name]()
    d = H.upload(w)
    y, mean, rstd, _ = H.gpu_fwd(d)
    dx, dsh, dsc, _ = H.gpu_bwd(d, mean, rstd)
    dx2 = t.empty_like(dx)
    dsh2, dsc2 = t.empty_like(dsh), t.empty_like(dsc)
    if w.dense is None:
        nb = A.adaln_bwd_varlen_recompute_workspace_size(w.R, w.nseg, w.nmod, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_bwd_varlen_recompute(d.dy, d.x, d.scale, dx2, dsh2, dsc2, d.cu, d.mod, w.nseg, w.R,
                                     w.nmod, w.D, H.EPS, ws, nb, w.dtype)
        assert A.adaln_read_status(ws) == 0
    else:
        Bt, N = w.dense
        nb = A.adaln_bwd_recompute_workspace_size(Bt, N, w.D, w.dtype)
        assert nb > A.adaln_bwd_workspace_size(Bt, N, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_bwd_recompute(d.dy, d.x, d.scale, dx2, dsh2, dsc2, ws, nb, Bt, N, w.D, H.EPS, w.dtype)
    t.cuda.synchronize()
    assert t.equal(dx, dx2)
    assert t.equal(dsh, dsh2) and t.equal(dsc, dsc2)
    del d, y, dx, dx2
    t.cuda.empty_cache()


@pytest.mark.parametrize("fill", [0x00, 0xFF, 0x5A])
def test_workspace_contents_do_not_matter(fill):
    """The backward's workspace needs no initialisation: zeroed, all-ones and patterned
    workspaces, reused call after call, give bitwise the results of a fresh one."""
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = synth.make("ws", 130, synth.BF16, 3072, [40, 3000, 1, 0, 9000, 513], [5, 0, 2, 2, 1, 0], 7,
                   x_mode=synth.ROWS_SCALED, dy_std=0.02)
    d = H.upload(w)
    _, mean, rstd, _ = H.gpu_fwd(d)
    ref = H.gpu_bwd(d, mean, rstd)[:3]
    nb = A.adaln_bwd_varlen_workspace_size(w.R, w.nseg, w.nmod, w.D, w.dtype)
    ws = t.full((nb,), fill, dtype=t.uint8, device="cuda")
    for _ in range(3):
        dx = t.empty_like(ref[0])
        dsh, dsc = t.empty_like(ref[1]), t.empty_like(ref[2])
        A.adaln_bwd_varlen(d.dy, d.x, mean, rstd, d.scale, dx, dsh, dsc, d.cu, d.mod, w.nseg, w.R,
                           w.nmod, w.D, ws, nb, w.dtype)
        assert A.adaln_read_status(ws) == 0
        assert t.equal(dx, ref[0]) and t.equal(dsh, ref[1]) and t.equal(dsc, ref[2])
