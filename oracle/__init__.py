"""TEST INFRASTRUCTURE ONLY: the CPU oracle for the fused AdaLN operator.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product (the CUDA library and its
binding) never does, and shares no code with it.

``adaln_oracle.cpp`` holds the operator (fp64, plain loops); ``bucket.py`` the
bucket-size rule. This module only compiles and marshals.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

from .bucket import bucket_batch  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adaln_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2


def compile_library(src: str, out: str) -> str:
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", tmp, src])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_library(_SRC, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    vp, i64, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_adaln_fwd.argtypes = [vp, vp, vp, ctypes.c_int, i64, vp, vp, i64, i64, i64, i64,
                                     dbl, vp, vp, vp]
    lib.oracle_adaln_fwd.restype = ctypes.c_int
    lib.oracle_adaln_bwd.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i64, vp, vp, i64, i64, i64,
                                     i64, vp, vp, vp]
    lib.oracle_adaln_bwd.restype = ctypes.c_int
    lib.oracle_round_to_bf16.argtypes = [vp, vp, i64]
    lib.oracle_round_to_bf16.restype = None
    return lib


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a test mutant)."""

    def __init__(self, path: Optional[str] = None):
        self.path = path or build()
        self.lib = _bind(self.path)

    def fwd(self, x, shift, scale, dtype, cu_seqlens, mod_idx, nmod, eps=1e-6,
            rows: Optional[tuple] = None):
        """Returns (y, mean, rstd) as float64 for rows [r0, r1) (default: all rows)."""
        D = x.shape[-1]
        cu, mod = _c(cu_seqlens, np.int64), _c(mod_idx, np.int64)
        r0, r1 = rows if rows is not None else (0, int(cu[-1]))
        x, shift, scale = _c(x), _c(shift), _c(scale)
        y = np.empty((r1 - r0, D), np.float64)
        mean = np.empty(r1 - r0, np.float64)
        rstd = np.empty(r1 - r0, np.float64)
        rc = self.lib.oracle_adaln_fwd(x.ctypes.data, shift.ctypes.data, scale.ctypes.data, dtype,
                                       D, cu.ctypes.data, mod.ctypes.data, len(mod), nmod, r0, r1,
                                       float(eps), y.ctypes.data, mean.ctypes.data,
                                       rstd.ctypes.data)
        if rc:
            raise ValueError("oracle_adaln_fwd rejected its arguments")
        return y, mean, rstd

    def bwd(self, dy, x, mean, rstd, scale, dtype, cu_seqlens, mod_idx, nmod,
            rows: Optional[tuple] = None, dshift=None, dscale=None):
        """Returns (dx, dshift, dscale) as float64. mean/rstd cover rows [r0, r1).
        dshift/dscale, if given ([nmod, D] float64), are accumulated into."""
        D = x.shape[-1]
        cu, mod = _c(cu_seqlens, np.int64), _c(mod_idx, np.int64)
        r0, r1 = rows if rows is not None else (0, int(cu[-1]))
        dy, x, scale = _c(dy), _c(x), _c(scale)
        mean, rstd = _c(mean, np.float64), _c(rstd, np.float64)
        assert mean.shape == (r1 - r0,) and rstd.shape == (r1 - r0,)
        dx = np.empty((r1 - r0, D), np.float64)
        if dshift is None:
            dshift = np.zeros((nmod, D), np.float64)
        if dscale is None:
            dscale = np.zeros((nmod, D), np.float64)
        assert dshift.dtype == np.float64 and dshift.flags.c_contiguous
        assert dscale.dtype == np.float64 and dscale.flags.c_contiguous
        rc = self.lib.oracle_adaln_bwd(dy.ctypes.data, x.ctypes.data, mean.ctypes.data,
                                       rstd.ctypes.data, scale.ctypes.data, dtype, D,
                                       cu.ctypes.data, mod.ctypes.data, len(mod), nmod, r0, r1,
                                       dx.ctypes.data, dshift.ctypes.data, dscale.ctypes.data)
        if rc:
            raise ValueError("oracle_adaln_bwd rejected its arguments")
        return dx, dshift, dscale

    def fwd_bwd_blocks(self, x, dy, shift, scale, dtype, cu_seqlens, mod_idx, nmod, rows, threads,
                       eps=1e-6, block_rows=1024):
        """Forward, then backward on the forward's statistics rounded to fp32 (as a caller that
        saves them in fp32 would), over rows [r0, r1), in blocks of `block_rows` rows spread over
        `threads` host threads (the library calls release the interpreter lock). Per-row
        outputs are discarded; returns the (dshift, dscale) sums. Used to time the oracle on
        all cores; each block is the plain per-row code above."""
        from concurrent.futures import ThreadPoolExecutor
        import threading

        r0, r1 = rows
        D = x.shape[-1]
        local = threading.local()
        accs = []
        lock = threading.Lock()

        def one(b0):
            b1 = min(r1, b0 + block_rows)
            if not hasattr(local, "acc"):
                local.acc = (np.zeros((nmod, D)), np.zeros((nmod, D)))
                with lock:
                    accs.append(local.acc)
            _, mean, rstd = self.fwd(x, shift, scale, dtype, cu_seqlens, mod_idx, nmod, eps=eps,
                                     rows=(b0, b1))
            self.bwd(dy, x, mean.astype(np.float32), rstd.astype(np.float32), scale, dtype, cu_seqlens,
                     mod_idx, nmod, rows=(b0, b1), dshift=local.acc[0], dscale=local.acc[1])

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(r0, r1, block_rows)))
        dsh = np.zeros((nmod, D))
        dsc = np.zeros((nmod, D))
        for a, b in accs:
            dsh += a
            dsc += b
        return dsh, dsc

    def round_bf16(self, v) -> np.ndarray:
        v = _c(np.asarray(v), np.float64)
        out = np.empty(v.shape, np.uint16)
        self.lib.oracle_round_to_bf16(v.ctypes.data, out.ctypes.data, v.size)
        return out


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
