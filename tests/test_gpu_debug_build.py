"""The index-checked debug build (libadaln_debug.so: the same sources with -DADALN_DEBUG, every
computed index of a global or shared-memory access checked against its buffer before the
access, a failed check recorded in a device word instead of trapping).

On the tiny workload and on odd shapes covering every staging mode and row form (plain
loads, bulk and copy rings, two rows a round, the wide and split forms, packed tables with
empty segments, the statistics-free and no-allocation backwards, the rank-order sum): no
check fails, the results are bitwise those of the release library, and the tiny workload
matches the oracle on every element.
"""
from __future__ import annotations

import contextlib

import numpy as np
import pytest

import synth
from tests import gpu_harness as H
from tests.test_gpu_parity import SMALL, _run_and_compare

pytestmark = pytest.mark.gpu

_DEBUG = {}


@pytest.fixture(scope="module")
def debug_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaln_layernorm_modulate_gb300 as A
    from adaln_layernorm_modulate_gb300 import build
    build.build(debug=True)  # built by the package build; rebuilt only if out of date
    release = A.lib()
    saved = (A.LIB_PATH, A._handle)
    A.LIB_PATH, A._handle = A.DEBUG_LIB_PATH, None
    try:
        _DEBUG["handle"] = A.lib()
    finally:
        A.LIB_PATH, A._handle = saved
    assert A._handle is release
    with library("debug") as AD:
        AD.adaln_debug_read(reset=True)
    yield _DEBUG["handle"]


@contextlib.contextmanager
def library(which: str):
    """Route the binding's calls to the debug or the release library for the block."""
    import adaln_layernorm_modulate_gb300 as A
    saved = (A.LIB_PATH, A._handle)
    if which == "debug":
        A.LIB_PATH, A._handle = A.DEBUG_LIB_PATH, _DEBUG["handle"]
    try:
        yield A
    finally:
        A.LIB_PATH, A._handle = saved


def _outputs(w):
    d = H.upload(w)
    y, mean, rstd, st = H.gpu_fwd(d)
    assert st == 0
    dx, dsh, dsc, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    return [H.to_host(y, w.dtype), H.to_host(mean, 0), H.to_host(rstd, 0), H.to_host(dx, w.dtype),
            H.to_host(dsh, 0), H.to_host(dsc, 0)]


ODD = {
    # N = 1 and N = 3 rows a sample, N = 257 (a ragged tail in every tile), one-warp rows.
    "dense-f32-3x1x128": lambda: synth.dense("dbg", 301, synth.F32, 3, 1, 128),
    "dense-bf16-1x3x1536": lambda: synth.dense("dbg", 302, synth.BF16, 1, 3, 1536),
    "dense-bf16-2x257x3072": lambda: synth.dense("dbg", 303, synth.BF16, 2, 257, 3072,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "dense-bf16-4x257x1536": lambda: synth.dense("dbg", 304, synth.BF16, 4, 257, 1536,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    # Widths the threads do not cover exactly (idle lanes, bounds on every vector).
    "packed-bf16-d264": SMALL["packed-bf16-d264"],
    "packed-f32-d128-many": SMALL["packed-f32-d128-many"],
    # Empty segments, shared and unused modulation rows.
    "packed-bf16-d3072-ragged": SMALL["packed-bf16-d3072-ragged"],
    # The copy ring, the wide form and the split form.
    "packed-bf16-d3072-copy-ring": SMALL["packed-bf16-d3072-copy-ring"],
    "packed-bf16-d16384-wide": SMALL["packed-bf16-d16384-wide"],
    "packed-f32-d15360-split": SMALL["packed-f32-d15360-split"],
    "dense-f32-2x21x16384": SMALL["dense-f32-2x21x16384"],
    # fp32 rows loaded straight into registers are gone; the widest bulk ring: fp32 D=14336.
    "dense-f32-2x19x14336": SMALL["dense-f32-2x19x14336"],
}


def test_tiny_workload_matches_the_oracle_under_the_debug_build(debug_lib, orc):
    with library("debug") as A:
        _run_and_compare(orc, synth.config(0))
        assert A.adaln_debug_read() == 0


@pytest.mark.parametrize("name", sorted(ODD))
def test_debug_build_checks_pass_and_match_the_release_build(debug_lib, name):
    w = ODD[name]()
    with library("release"):
        ref = _outputs(w)
    with library("debug") as A:
        got = _outputs(w)
        word = A.adaln_debug_read(reset=True)
    assert word == 0, {v: n for v, n in A.DEBUG_CLASSES.items() if word & v}
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


def test_debug_build_recompute_noalloc_and_rank_sum(debug_lib):
    t = H.torch()
    w = SMALL["dense-bf16-2x300x1536"]()
    Bt, N = w.dense
    results = {}
    for which in ("release", "debug"):
        with library(which) as A:
            d = H.upload(w)
            dx = t.empty((w.R, w.D), dtype=H.torch_dtype(w.dtype), device="cuda")
            dsh = t.empty((w.nmod, w.D), dtype=t.float32, device="cuda")
            dsc = t.empty_like(dsh)
            nb = A.adaln_bwd_recompute_workspace_size(Bt, N, w.D, w.dtype)
            ws = t.empty(nb, dtype=t.uint8, device="cuda")
            A.adaln_bwd_recompute(d.dy, d.x, d.scale, dx, dsh, dsc, ws, nb, Bt, N, w.D, H.EPS, w.dtype)
            assert A.adaln_read_status(ws) == 0
            _, mean, rstd, _ = H.gpu_fwd(d)
            dx2, dsh2, dsc2 = t.empty_like(dx), t.empty_like(dsh), t.empty_like(dsc)
            A.adaln_bwd_noalloc(d.dy, d.x, mean, rstd, d.scale, dx2, dsh2, dsc2, Bt, N, w.D, w.dtype)
            assert A.adaln_noalloc_read_status() == 0
            parts = t.from_numpy(np.random.default_rng(7).standard_normal((3, 5 * 257 + 3))
                                 .astype(np.float32)).cuda()
            out = t.empty(parts.shape[1], device="cuda")
            A.adaln_sum_ranks(parts, out, 3, parts.shape[1])
            results[which] = [H.to_host(v, w.dtype if i in (0, 3) else 0)
                              for i, v in enumerate((dx, dsh, dsc, dx2, dsh2, dsc2))] + [out.cpu().numpy()]
            if which == "debug":
                assert A.adaln_debug_read(reset=True) == 0
    for a, b in zip(results["release"], results["debug"]):
        assert np.array_equal(a, b)
