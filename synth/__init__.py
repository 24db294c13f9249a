"""Seeded synthetic workloads for the fused AdaLN operator.

Shared by the CPU oracle side and the CUDA side, and by nothing else: it draws
random inputs (``synth.c``: counter-based SplitMix64 + Box-Muller in double,
rounded once to the I/O dtype) and lays out the packed row tables. It contains
none of the operator's arithmetic.

The workloads mirror the video-DiT / MMDiT shapes of the AdaptiveLoad paper
(technical summary, section 4 "Experimental results": Wan 2.1 trained on a
mixed-length corpus). The corpus itself is not available; the value
distributions below stand in for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

F32, BF16, F64 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F64: "f64"}
NP_STORAGE = {F32: np.float32, BF16: np.uint16, F64: np.float64}

ROWS_NORMAL, ROWS_SCALED, ROWS_ADVERSARIAL = 0, 1, 2

# One stream id per tensor role; a role's draws never overlap another's.
STREAM_X, STREAM_DY, STREAM_SHIFT, STREAM_SCALE = 1, 2, 3, 4

_lib_handle = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so beside it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal.argtypes = [u64, u64, i64, dbl, dbl, ctypes.c_int, vp]
        lib.synth_normal.restype = ctypes.c_int
        lib.synth_rows.argtypes = [u64, u64, ctypes.c_int, vp, i64, i64, dbl, dbl, ctypes.c_int, vp]
        lib.synth_rows.restype = ctypes.c_int
        lib.synth_round_bf16.argtypes = [vp, vp, i64]
        lib.synth_round_bf16.restype = None
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, stream: int, n: int, mean: float, std: float, dtype: int) -> np.ndarray:
    out = np.empty(n, dtype=NP_STORAGE[dtype])
    rc = _lib().synth_normal(seed, stream, n, mean, std, dtype, _ptr(out))
    if rc:
        raise ValueError("synth_normal rejected its arguments")
    return out


def rows(seed: int, stream: int, mode: int, cu_seqlens: np.ndarray, D: int, dtype: int,
         mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    R = int(cu[-1])
    out = np.empty((R, D), dtype=NP_STORAGE[dtype])
    rc = _lib().synth_rows(seed, stream, mode, _ptr(cu), len(cu) - 1, D, mean, std, dtype, _ptr(out))
    if rc:
        raise ValueError("synth_rows rejected its arguments")
    return out


def round_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _lib().synth_round_bf16(_ptr(v), _ptr(out), v.size)
    return out


def widen(a: np.ndarray, dtype: int) -> np.ndarray:
    """Exact value of stored elements as float64 (bf16 bits -> double)."""
    if dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


@dataclass
class Workload:
    """A packed AdaLN problem: R rows of width D, split into segments, each segment
    modulated by one row of the [nmod, D] shift/scale tables."""
    name: str
    seed: int
    dtype: int
    D: int
    cu_seqlens: np.ndarray          # int64 [nseg + 1]
    mod_idx: np.ndarray             # int64 [nseg]
    nmod: int
    dense: Optional[tuple] = None   # (Bt, N) when the layout is a dense [Bt, N, D] batch
    x: Optional[np.ndarray] = None  # storage dtype, [R, D]
    dy: Optional[np.ndarray] = None
    shift: Optional[np.ndarray] = None  # [nmod, D]
    scale: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def nseg(self) -> int:
        return len(self.mod_idx)


def make(name: str, seed: int, dtype: int, D: int, seg_lens: Sequence[int],
         mod_idx: Optional[Sequence[int]] = None, nmod: Optional[int] = None,
         x_mode: int = ROWS_NORMAL, x_mean: float = 0.0, x_std: float = 1.0,
         mod_std: float = 0.1, dy_std: float = 1.0, dense: Optional[tuple] = None,
         generate: bool = True) -> Workload:
    lens = np.asarray(list(seg_lens), dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    if mod_idx is None:
        mod_idx = np.arange(len(lens), dtype=np.int64)
    mod = np.asarray(list(mod_idx), dtype=np.int64)
    if nmod is None:
        nmod = int(mod.max()) + 1 if len(mod) else 0
    w = Workload(name=name, seed=seed, dtype=dtype, D=D, cu_seqlens=cu, mod_idx=mod, nmod=nmod,
                 dense=dense)
    w.meta = dict(x_mode=x_mode, x_mean=x_mean, x_std=x_std, mod_std=mod_std, dy_std=dy_std)
    if generate:
        fill(w)
    return w


def fill(w: Workload) -> Workload:
    m = w.meta
    w.x = rows(w.seed, STREAM_X, m["x_mode"], w.cu_seqlens, w.D, w.dtype, m["x_mean"], m["x_std"])
    w.dy = normal(w.seed, STREAM_DY, w.R * w.D, 0.0, m["dy_std"], w.dtype).reshape(w.R, w.D)
    w.shift = normal(w.seed, STREAM_SHIFT, w.nmod * w.D, 0.0, m["mod_std"], w.dtype).reshape(w.nmod, w.D)
    w.scale = normal(w.seed, STREAM_SCALE, w.nmod * w.D, 0.0, m["mod_std"], w.dtype).reshape(w.nmod, w.D)
    return w


def dense(name: str, seed: int, dtype: int, Bt: int, N: int, D: int, **kw) -> Workload:
    return make(name, seed, dtype, D, [N] * Bt, list(range(Bt)), Bt, dense=(Bt, N), **kw)


# ---------------------------------------------------------------------------------------
# The five workloads. Index = seed.
# ---------------------------------------------------------------------------------------
BUCKET_S = (256, 1024, 4096, 16384, 32760, 75600)
BUCKET_M_MEM = 131072
BUCKET_M_COMP = 131072 * 4096
BUCKET_P = 2
MMDIT_TEXT_N, MMDIT_VIDEO_N = 512, 32760


def bucket(S: int, bucket_batch: Callable[[int, int, int, int], int], generate: bool = True) -> Workload:
    """One bucket of workload 3 as its own packed call: bucket_batch(S, ...) segments of
    length S, bf16, D=3072, one modulation row per segment, x and dy as workload 1."""
    B = int(bucket_batch(S, BUCKET_M_MEM, BUCKET_M_COMP, BUCKET_P))
    w = make("bucket-s%d-bf16-d3072-%dseg" % (S, B), 3, BF16, 3072, [S] * B,
             x_mode=ROWS_SCALED, mod_std=0.1, dy_std=0.02, generate=generate)
    w.meta["batches"] = [B]
    w.meta["bucket_s"] = [S]
    return w


def config(idx: int, bucket_batch: Optional[Callable[[int, int, int, int], int]] = None,
           dtype: Optional[int] = None, generate: bool = True) -> Workload:
    """Build workload `idx` (0..4).

    0  tiny dense fp32 x[2,256,128]
    1  Wan-2.1-1.3B width, bf16 x[1,32760,1536] (21x30x52 latent tokens)
    2  Wan-2.1-14B width, bf16 x[1,32760,5120]
    3  packed mixed-length buckets, bf16, D=3072: per length S the bucket holds
       bucket_batch(S, 131072, 131072*4096, 2) segments (the caller supplies the rule)
    4  MMDiT dual stream, D=3072, Bt=2, text 512 + video 32760 tokens, adversarial rows;
       dtype f32 (default) or bf16
    """
    if idx == 0:
        return dense("tiny-f32-2x256x128", 0, F32, 2, 256, 128, x_mode=ROWS_NORMAL,
                     mod_std=0.1, dy_std=1.0, generate=generate)
    if idx in (1, 2):
        D = 1536 if idx == 1 else 5120
        return dense("wan-%s-bf16-1x32760x%d" % ("1.3b" if idx == 1 else "14b", D), idx, BF16,
                     1, 32760, D, x_mode=ROWS_SCALED, mod_std=0.1, dy_std=0.02, generate=generate)
    if idx == 3:
        if bucket_batch is None:
            raise ValueError("workload 3 needs the bucket-size rule")
        lens, batches = [], []
        for S in BUCKET_S:
            B = int(bucket_batch(S, BUCKET_M_MEM, BUCKET_M_COMP, BUCKET_P))
            batches.append(B)
            lens += [S] * B
        w = make("varlen-bf16-d3072-%dseg" % len(lens), 3, BF16, 3072, lens,
                 x_mode=ROWS_SCALED, mod_std=0.1, dy_std=0.02, generate=generate)
        w.meta["batches"] = batches
        w.meta["bucket_s"] = list(BUCKET_S)
        return w
    if idx == 4:
        dt = F32 if dtype is None else dtype
        T, V = MMDIT_TEXT_N, MMDIT_VIDEO_N
        # table rows: [text b0, text b1, video b0, video b1]; packed order b0-text, b0-video,
        # b1-text, b1-video
        w = make("mmdit-%s-d3072-2x(512+32760)" % DTYPE_NAMES[dt], 4, dt, 3072, [T, V, T, V],
                 [0, 2, 1, 3], 4, x_mode=ROWS_ADVERSARIAL, mod_std=0.5, dy_std=0.02,
                 generate=generate)
        return w
    raise ValueError("no workload %r" % idx)
