"""Test-side helpers: run the CUDA path through the C-ABI binding on device copies of a
synthetic workload, run the oracle on the same host bits, and compare with the
tolerances of the operator's parity bar:

  fp32 I/O: y, dx within 1e-5 * max(1, |ref|) elementwise; dshift, dscale within a
            relative L2 error of 1e-5.
  bf16 I/O: y, dx within 1 bf16 ulp of the oracle rounded (once, RNE) to bf16, plus 1e-3;
            the fp32 dshift, dscale within a relative L2 error of 1e-3.
  statistics (fp32 always): mean within 1e-5 * max(1, |mean|, std), rstd relative 1e-5.
"""
from __future__ import annotations

import os
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional

import numpy as np

import synth

EPS = float(np.float32(1e-6))


def torch():
    import torch as t
    return t


def to_dev(a: np.ndarray, dtype: int, device="cuda"):
    """Host storage array -> device tensor with the same bits."""
    t = torch()
    if dtype == synth.BF16:
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.bfloat16).to(device)
    return t.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(tensor, dtype: int) -> np.ndarray:
    t = torch()
    tensor = tensor.detach().cpu().contiguous()
    if tensor.dtype == t.bfloat16:
        return tensor.view(t.int16).numpy().view(np.uint16)
    return tensor.numpy()


def torch_dtype(dtype: int):
    t = torch()
    return t.bfloat16 if dtype == synth.BF16 else t.float32


@dataclass
class DevWorkload:
    w: synth.Workload
    x: object
    dy: object
    shift: object
    scale: object
    cu: object
    mod: object


def upload(w: synth.Workload) -> DevWorkload:
    t = torch()
    cu = t.from_numpy(w.cu_seqlens.astype(np.int32)).cuda()
    mod = t.from_numpy(w.mod_idx.astype(np.int32)).cuda() if w.nseg else t.zeros(1, dtype=t.int32).cuda()
    return DevWorkload(w, to_dev(w.x, w.dtype), to_dev(w.dy, w.dtype), to_dev(w.shift, w.dtype),
                       to_dev(w.scale, w.dtype), cu, mod)


@dataclass
class GpuOut:
    y: object
    mean: object
    rstd: object
    dx: Optional[object] = None
    dshift: Optional[object] = None
    dscale: Optional[object] = None
    status_fwd: int = 0
    status_bwd: int = 0


def gpu_fwd(d: DevWorkload, packed: Optional[bool] = None):
    import adaln_layernorm_modulate_gb300 as A
    t = torch()
    w = d.w
    packed = (w.dense is None) if packed is None else packed
    y = t.empty((w.R, w.D), dtype=torch_dtype(w.dtype), device="cuda")
    mean = t.empty(w.R, dtype=t.float32, device="cuda")
    rstd = t.empty(w.R, dtype=t.float32, device="cuda")
    status = 0
    if packed:
        nb = A.adaln_fwd_varlen_workspace_size(w.R, w.nseg, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_fwd_varlen(d.x, d.shift, d.scale, y, mean, rstd, d.cu, d.mod, w.nseg, w.R, w.nmod,
                           w.D, EPS, ws, nb, w.dtype)
        status = A.adaln_read_status(ws)
    else:
        Bt, N = w.dense
        A.adaln_fwd(d.x, d.shift, d.scale, y, mean, rstd, Bt, N, w.D, EPS, w.dtype)
    return y, mean, rstd, status


def gpu_bwd(d: DevWorkload, mean, rstd, packed: Optional[bool] = None):
    import adaln_layernorm_modulate_gb300 as A
    t = torch()
    w = d.w
    packed = (w.dense is None) if packed is None else packed
    dx = t.empty((w.R, w.D), dtype=torch_dtype(w.dtype), device="cuda")
    dshift = t.empty((w.nmod, w.D), dtype=t.float32, device="cuda")
    dscale = t.empty((w.nmod, w.D), dtype=t.float32, device="cuda")
    if packed:
        nb = A.adaln_bwd_varlen_workspace_size(w.R, w.nseg, w.nmod, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_bwd_varlen(d.dy, d.x, mean, rstd, d.scale, dx, dshift, dscale, d.cu, d.mod, w.nseg,
                           w.R, w.nmod, w.D, ws, nb, w.dtype)
    else:
        Bt, N = w.dense
        nb = A.adaln_bwd_workspace_size(Bt, N, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_bwd(d.dy, d.x, mean, rstd, d.scale, dx, dshift, dscale, ws, nb, Bt, N, w.D, w.dtype)
    status = A.adaln_read_status(ws)
    return dx, dshift, dscale, status


# ------------------------------------------------------------------------------------------
# comparisons
# ------------------------------------------------------------------------------------------
# ulp of a bf16 value by its 8-bit exponent field e: 2^(e-134) for normal values (8
# significant bits in the binade [2^(e-127), 2^(e-126))), and the smallest subnormal 2^-133
# for zeros and subnormals.
_BF16_ULP_BY_EXPONENT = np.array([2.0 ** -133] + [2.0 ** (e - 134) for e in range(1, 256)])


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    return _BF16_ULP_BY_EXPONENT[(np.asarray(bits, dtype=np.uint16) >> 7) & 0xFF]


def check_io(gpu: np.ndarray, ref: np.ndarray, dtype: int, orc, what: str, extra=None):
    """Elementwise I/O-tensor check. gpu: storage dtype array; ref: float64."""
    if dtype == synth.BF16:
        rb = orc.round_bf16(ref)
        tol = bf16_ulp(rb) + 1e-3
        diff = np.abs(synth.widen(gpu, synth.BF16) - synth.widen(rb, synth.BF16))
    else:
        tol = 1e-5 * np.maximum(1.0, np.abs(ref))
        diff = np.abs(gpu.astype(np.float64) - ref)
    if extra is not None:
        tol = tol + extra
    bad = diff > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements out of tolerance; first %s: gpu-ref diff %s tol %s"
                             % (what, int(bad.sum()), bad.size, idx.tolist(),
                                diff[bad][:5].tolist(), tol[bad][:5].tolist()))


def check_stats(mean_gpu, rstd_gpu, mean_ref, rstd_ref, what="stats"):
    mean_gpu = mean_gpu.astype(np.float64)
    rstd_gpu = rstd_gpu.astype(np.float64)
    # fp32 sums of a row carry errors relative to the row's spread as well as its mean.
    spread = 1.0 / np.maximum(rstd_ref, 1e-300)
    bad_m = np.abs(mean_gpu - mean_ref) > 1e-5 * np.maximum(np.maximum(1.0, np.abs(mean_ref)), spread)
    bad_r = np.abs(rstd_gpu - rstd_ref) > 1e-5 * np.abs(rstd_ref)
    assert not bad_m.any(), "%s: mean out of tolerance at rows %s" % (what, np.argwhere(bad_m)[:5].ravel())
    assert not bad_r.any(), "%s: rstd out of tolerance at rows %s" % (what, np.argwhere(bad_r)[:5].ravel())


def rel_l2(gpu: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm(gpu.astype(np.float64).ravel() - ref.ravel())
    return float(num / den) if den > 0 else float(num)


def grad_tol(dtype: int) -> float:
    return 1e-3 if dtype == synth.BF16 else 1e-5


def round_f32(a: np.ndarray) -> np.ndarray:
    return a.astype(np.float32).astype(np.float64)


def stat_shift_bound(ref_dx_terms):
    """Extra dx tolerance for a pipeline test: the GPU backward consumes the GPU's own fp32
    statistics, which may sit one fp32 ulp from the oracle's rounded ones. A mean shift of
    dm moves xhat by rstd*dm on the whole row and dx by at most
    rstd^2 * dm * (|mean(g*xhat)| + |xhat| * |mean(g)|); rstd's own ulp is covered by the
    relative tolerance."""
    rstd, mean, xhat, mg, mgx = ref_dx_terms
    dm = np.spacing(np.abs(mean).astype(np.float32)).astype(np.float64)
    return (rstd * rstd * dm)[:, None] * (np.abs(mgx)[:, None] + np.abs(xhat) * np.abs(mg)[:, None]) * 1.01


# ------------------------------------------------------------------------------------------
# every row of a large workload against the oracle
# ------------------------------------------------------------------------------------------
CHUNK_ELEMENTS = 1 << 23  # elements of a row chunk (64 MB per float64 array)


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def row_chunks(R: int, D: int):
    n = max(1, CHUNK_ELEMENTS // D)
    return [(a, min(R, a + n)) for a in range(0, R, n)]


def mod_of_rows(w, r0: int, r1: int) -> np.ndarray:
    seg = np.searchsorted(w.cu_seqlens, np.arange(r0, r1), side="right") - 1
    return np.asarray(w.mod_idx)[seg]


def dx_terms(w, mean, rstd, rows):
    """Oracle-side quantities of rows [r0, r1) for stat_shift_bound."""
    r0, r1 = rows
    x = synth.widen(w.x[r0:r1], w.dtype)
    dy = synth.widen(w.dy[r0:r1], w.dtype)
    g = dy * (1 + synth.widen(w.scale, w.dtype)[mod_of_rows(w, r0, r1)])
    xhat = (x - mean[:, None]) * rstd[:, None]
    return rstd, mean, xhat, g.mean(axis=1), (g * xhat).mean(axis=1)


def forward_all_rows(orc, w, y_h, mean_h, rstd_h, what=""):
    """Every row of y, mean, rstd (host copies of the GPU outputs) against the oracle, a chunk
    of rows at a time on a thread pool. Returns the oracle's statistics rounded to fp32 (as
    float64 arrays), which the backward checks consume."""
    m32 = np.empty(w.R)
    r32 = np.empty(w.R)

    def one(rows):
        r0, r1 = rows
        ry, rmean, rrstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod,
                                   eps=EPS, rows=rows)
        check_io(y_h[r0:r1], ry, w.dtype, orc, "%sy rows %d:%d" % (what, r0, r1))
        check_stats(mean_h[r0:r1], rstd_h[r0:r1], rmean, rrstd, "%sstats rows %d:%d" % (what, r0, r1))
        m32[r0:r1] = round_f32(rmean)
        r32[r0:r1] = round_f32(rrstd)

    with ThreadPoolExecutor(workers()) as ex:
        list(ex.map(one, row_chunks(w.R, w.D)))
    return m32, r32


def backward_all_rows(orc, w, m32, r32, pipeline=None, isolated=None, what=""):
    """Every row of dx and every row of dshift/dscale against the oracle's backward on the
    oracle's fp32-rounded statistics (m32, r32). `isolated` = host (dx, dshift, dscale) of a
    GPU backward that consumed those same statistics: strict tolerance. `pipeline` = host
    (dx, dshift, dscale) of a GPU backward that consumed the GPU forward's own statistics:
    dx gets the one-ulp mean-shift bound on top. dshift/dscale are checked row by row
    (relative L2), and rows of the modulation table that no token uses must be exactly 0."""
    lock = threading.Lock()
    accs = []
    local = threading.local()

    def one(rows):
        r0, r1 = rows
        if not hasattr(local, "acc"):
            local.acc = (np.zeros((w.nmod, w.D)), np.zeros((w.nmod, w.D)))
            with lock:
                accs.append(local.acc)
        rdx, _, _ = orc.bwd(w.dy, w.x, m32[r0:r1], r32[r0:r1], w.scale, w.dtype, w.cu_seqlens,
                            w.mod_idx, w.nmod, rows=rows, dshift=local.acc[0], dscale=local.acc[1])
        if isolated is not None:
            check_io(isolated[0][r0:r1], rdx, w.dtype, orc, "%sdx (isolated) rows %d:%d" % (what, r0, r1))
        if pipeline is not None:
            extra = stat_shift_bound(dx_terms(w, m32[r0:r1], r32[r0:r1], rows))
            check_io(pipeline[0][r0:r1], rdx, w.dtype, orc, "%sdx (pipeline) rows %d:%d" % (what, r0, r1),
                     extra=extra)

    with ThreadPoolExecutor(workers()) as ex:
        list(ex.map(one, row_chunks(w.R, w.D)))
    ref_sh = np.zeros((w.nmod, w.D))
    ref_sc = np.zeros((w.nmod, w.D))
    for a_sh, a_sc in accs:
        ref_sh += a_sh
        ref_sc += a_sc
    used = np.zeros(w.nmod, bool)
    used[np.asarray(w.mod_idx)[np.diff(w.cu_seqlens) > 0]] = True
    tol = grad_tol(w.dtype)
    for label, got in (("isolated", isolated), ("pipeline", pipeline)):
        if got is None:
            continue
        for name, g, ref in (("dshift", got[1], ref_sh), ("dscale", got[2], ref_sc)):
            assert np.all(g[~used] == 0), "%s%s (%s): unused modulation rows not zero" % (what, name, label)
            assert rel_l2(g, ref) <= tol, "%s%s (%s): whole table" % (what, name, label)
            for m in np.nonzero(used)[0]:
                e = rel_l2(g[m], ref[m])
                assert e <= tol, "%s%s (%s) row %d: relative L2 %.3g" % (what, name, label, m, e)
    return ref_sh, ref_sc
