"""Thin Python binding of libadaln (fused AdaLN forward/backward for GB300, sm_103a).

Every function has the name and argument order of its C counterpart in
``include/adaln.h`` and only marshals arguments: device buffers may be given as
torch tensors (their ``data_ptr()`` is passed) or as raw integer addresses;
``stream`` may be a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None
for torch's current stream. Every step of the computation runs in the library's
CUDA kernels. A nonzero status raises :class:`AdalnError` (``adaln_read_status``
returns it instead).

The library is built in-tree by ``build.build()``. It is loaded on first use; if it
is missing, that first call raises ImportError — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Any

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libadaln.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libadaln_debug.so")  # build(debug=True): index-checked kernels

ADALN_F32, ADALN_BF16 = 0, 1
STATUS = {
    0: "ADALN_OK", 1: "ADALN_ERR_INVALID_ARG", 2: "ADALN_ERR_UNSUPPORTED",
    3: "ADALN_ERR_ALIGNMENT", 4: "ADALN_ERR_WORKSPACE", 5: "ADALN_ERR_CUDA",
    6: "ADALN_ERR_BAD_SEQLENS", 7: "ADALN_ERR_BAD_MOD_IDX", 8: "ADALN_ERR_TIMEOUT",
}
EXPORTS = (
    "adaln_fwd", "adaln_bwd_workspace_size", "adaln_bwd", "adaln_bwd_partials", "adaln_bwd_reduce",
    "adaln_fwd_varlen_workspace_size", "adaln_fwd_varlen", "adaln_bwd_varlen_workspace_size",
    "adaln_bwd_varlen", "adaln_bwd_varlen_partials", "adaln_bwd_varlen_reduce",
    "adaln_read_status", "adaln_bwd_recompute_workspace_size", "adaln_bwd_recompute",
    "adaln_bwd_varlen_recompute_workspace_size", "adaln_bwd_varlen_recompute", "adaln_bwd_noalloc", "adaln_noalloc_read_status", "adaln_sum_ranks", "adaln_debug_read",
    "adaln_bucket_batch", "adaln_bucket_batch_real",
    "adaln_fit_step_cost", "adaln_bucket_load_cv", "adaln_status_string",
)
NOALLOC_SCRATCH_BYTES = 16 << 20  # ADALN_NOALLOC_SCRATCH_BYTES


class AdalnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, _status_text(status)))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libadaln.so is not built (%s); run "
                          "adaln_layernorm_modulate_gb300.build.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                             ctypes.c_size_t)
    ci = ctypes.c_int
    sig = {
        "adaln_fwd": ([vp, vp, vp, vp, vp, vp, i64, i64, i64, f32, ci, vp], ci),
        "adaln_bwd_workspace_size": ([i64, i64, i64, ci], sz),
        "adaln_bwd": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, i64, ci, vp], ci),
        "adaln_bwd_partials": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, i64, ci, vp], ci),
        "adaln_bwd_reduce": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, i64, ci, vp], ci),
        "adaln_fwd_varlen_workspace_size": ([i64, i32, i64, ci], sz),
        "adaln_fwd_varlen": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, f32, vp, sz,
                              ci, vp], ci),
        "adaln_bwd_varlen_workspace_size": ([i64, i32, i64, i64, ci], sz),
        "adaln_bwd_varlen": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, vp,
                              sz, ci, vp], ci),
        "adaln_bwd_varlen_partials": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64,
                                       vp, sz, ci, vp], ci),
        "adaln_bwd_varlen_reduce": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64,
                                     vp, sz, ci, vp], ci),
        "adaln_read_status": ([vp, vp], ci),
        "adaln_bwd_recompute_workspace_size": ([i64, i64, i64, ci], sz),
        "adaln_bwd_recompute": ([vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, i64, f32, ci, vp], ci),
        "adaln_bwd_varlen_recompute_workspace_size": ([i64, i32, i64, i64, ci], sz),
        "adaln_bwd_varlen_recompute": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, f32, vp,
                                        sz, ci, vp], ci),
        "adaln_bwd_noalloc": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, vp], ci),
        "adaln_noalloc_read_status": ([vp], ci),
        "adaln_sum_ranks": ([vp, vp, i32, i64, vp], ci),
        "adaln_debug_read": ([vp, ci], ci),
        "adaln_bucket_batch": ([i64, i64, i64, i32], i64),
        "adaln_bucket_batch_real": ([i64, i64, i64, ctypes.c_double], i64),
        "adaln_fit_step_cost": ([vp, vp, vp, i64, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_double, vp], ci),
        "adaln_bucket_load_cv": ([vp, i64, vp, i32, i64, i64, ctypes.c_double, i32, vp], ci),
        "adaln_status_string": ([ci], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_handle = None


def lib() -> ctypes.CDLL:
    """The loaded libadaln (loads it on first use; raises ImportError if not built)."""
    global _handle
    if _handle is None:
        _handle = _load()
    return _handle


def _status_text(status: int) -> str:
    return lib().adaln_status_string(int(status)).decode()


def _ptr(t: Any) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(s: Any) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _dtype(dtype: Any, t: Any) -> int:
    if dtype is None:
        import torch
        if t.dtype == torch.bfloat16:
            return ADALN_BF16
        if t.dtype == torch.float32:
            return ADALN_F32
        raise TypeError("unsupported tensor dtype %s" % t.dtype)
    return int(dtype)


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise AdalnError(fn, status)


def adaln_fwd(x, shift, scale, y, mean, rstd, Bt, N, D, eps=1e-6, dtype=None, stream=None):
    _check("adaln_fwd", lib().adaln_fwd(_ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(mean),
                                       _ptr(rstd), Bt, N, D, eps, _dtype(dtype, x),
                                       _stream(stream)))


def adaln_bwd_workspace_size(Bt, N, D, dtype) -> int:
    return int(lib().adaln_bwd_workspace_size(Bt, N, D, int(dtype)))


def adaln_bwd(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes, Bt, N, D,
              dtype=None, stream=None):
    _check("adaln_bwd", lib().adaln_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale),
                                       _ptr(dx), _ptr(dshift), _ptr(dscale), _ptr(workspace),
                                       workspace_bytes, Bt, N, D, _dtype(dtype, dy),
                                       _stream(stream)))


def adaln_bwd_partials(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes,
                       Bt, N, D, dtype=None, stream=None):
    _check("adaln_bwd_partials", lib().adaln_bwd_partials(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), _ptr(workspace), workspace_bytes, Bt, N, D, _dtype(dtype, dy),
        _stream(stream)))


def adaln_bwd_reduce(dy, x, mean, rstd, scale, dx, dshift, dscale, workspace, workspace_bytes,
                     Bt, N, D, dtype=None, stream=None):
    _check("adaln_bwd_reduce", lib().adaln_bwd_reduce(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), _ptr(workspace), workspace_bytes, Bt, N, D, _dtype(dtype, dy),
        _stream(stream)))


def adaln_fwd_varlen_workspace_size(total_tokens, nseg, D, dtype) -> int:
    return int(lib().adaln_fwd_varlen_workspace_size(total_tokens, nseg, D, int(dtype)))


def adaln_fwd_varlen(x, shift, scale, y, mean, rstd, cu_seqlens, mod_idx, nseg, total_tokens,
                     nmod, D, eps, workspace, workspace_bytes, dtype=None, stream=None):
    _check("adaln_fwd_varlen", lib().adaln_fwd_varlen(
        _ptr(x), _ptr(shift), _ptr(scale), _ptr(y), _ptr(mean), _ptr(rstd), _ptr(cu_seqlens),
        _ptr(mod_idx), nseg, total_tokens, nmod, D, eps, _ptr(workspace), workspace_bytes,
        _dtype(dtype, x), _stream(stream)))


def adaln_bwd_varlen_workspace_size(total_tokens, nseg, nmod, D, dtype) -> int:
    return int(lib().adaln_bwd_varlen_workspace_size(total_tokens, nseg, nmod, D, int(dtype)))


def adaln_bwd_varlen(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx, nseg,
                     total_tokens, nmod, D, workspace, workspace_bytes, dtype=None, stream=None):
    _check("adaln_bwd_varlen", lib().adaln_bwd_varlen(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), _ptr(cu_seqlens), _ptr(mod_idx), nseg, total_tokens, nmod, D,
        _ptr(workspace), workspace_bytes, _dtype(dtype, dy), _stream(stream)))


def adaln_bwd_varlen_partials(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx,
                              nseg, total_tokens, nmod, D, workspace, workspace_bytes, dtype=None,
                              stream=None):
    _check("adaln_bwd_varlen_partials", lib().adaln_bwd_varlen_partials(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), _ptr(cu_seqlens), _ptr(mod_idx), nseg, total_tokens, nmod, D,
        _ptr(workspace), workspace_bytes, _dtype(dtype, dy), _stream(stream)))


def adaln_bwd_varlen_reduce(dy, x, mean, rstd, scale, dx, dshift, dscale, cu_seqlens, mod_idx,
                            nseg, total_tokens, nmod, D, workspace, workspace_bytes, dtype=None,
                            stream=None):
    _check("adaln_bwd_varlen_reduce", lib().adaln_bwd_varlen_reduce(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), _ptr(cu_seqlens), _ptr(mod_idx), nseg, total_tokens, nmod, D,
        _ptr(workspace), workspace_bytes, _dtype(dtype, dy), _stream(stream)))


def adaln_bwd_recompute_workspace_size(Bt, N, D, dtype) -> int:
    return int(lib().adaln_bwd_recompute_workspace_size(Bt, N, D, int(dtype)))


def adaln_bwd_recompute(dy, x, scale, dx, dshift, dscale, workspace, workspace_bytes, Bt, N, D,
                        eps=1e-6, dtype=None, stream=None):
    _check("adaln_bwd_recompute", lib().adaln_bwd_recompute(
        _ptr(dy), _ptr(x), _ptr(scale), _ptr(dx), _ptr(dshift), _ptr(dscale), _ptr(workspace),
        workspace_bytes, Bt, N, D, eps, _dtype(dtype, x), _stream(stream)))


def adaln_bwd_varlen_recompute_workspace_size(total_tokens, nseg, nmod, D, dtype) -> int:
    return int(lib().adaln_bwd_varlen_recompute_workspace_size(total_tokens, nseg, nmod, D, int(dtype)))


def adaln_bwd_varlen_recompute(dy, x, scale, dx, dshift, dscale, cu_seqlens, mod_idx, nseg,
                               total_tokens, nmod, D, eps, workspace, workspace_bytes, dtype=None,
                               stream=None):
    _check("adaln_bwd_varlen_recompute", lib().adaln_bwd_varlen_recompute(
        _ptr(dy), _ptr(x), _ptr(scale), _ptr(dx), _ptr(dshift), _ptr(dscale), _ptr(cu_seqlens),
        _ptr(mod_idx), nseg, total_tokens, nmod, D, eps, _ptr(workspace), workspace_bytes,
        _dtype(dtype, x), _stream(stream)))


def adaln_read_status(workspace, stream=None) -> int:
    return int(lib().adaln_read_status(_ptr(workspace), _stream(stream)))


def adaln_bwd_noalloc(dy, x, mean, rstd, scale, dx, dshift, dscale, Bt, N, D, dtype=None,
                      stream=None):
    """adaln_bwd without a workspace, for callers that cannot allocate device memory; its
    scratch is a fixed array inside the library (see include/adaln.h)."""
    _check("adaln_bwd_noalloc", lib().adaln_bwd_noalloc(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(scale), _ptr(dx), _ptr(dshift),
        _ptr(dscale), Bt, N, D, _dtype(dtype, dy), _stream(stream)))


def adaln_noalloc_read_status(stream=None) -> int:
    return int(lib().adaln_noalloc_read_status(_stream(stream)))


def adaln_sum_ranks(parts, out, world, n, stream=None):
    """out[i] = parts[0][i] + ... + parts[world - 1][i], added in rank order (device fp32)."""
    _check("adaln_sum_ranks", lib().adaln_sum_ranks(_ptr(parts), _ptr(out), world, n, _stream(stream)))


DEBUG_CLASSES = {1: "rows", 2: "stats", 4: "mod", 8: "partials", 16: "segments", 32: "shared",
                 64: "grads", 128: "ranks", 256: "status"}  # ADALN_DEBUG_* bits


def adaln_debug_read(reset=False) -> int:
    """The debug build's word of failed index checks since the last reset (0: none); raises
    AdalnError (ADALN_ERR_UNSUPPORTED) on the release build."""
    word = ctypes.c_uint32(0)
    _check("adaln_debug_read", lib().adaln_debug_read(ctypes.addressof(word), 1 if reset else 0))
    return int(word.value)


def adaln_bucket_batch(S, M_mem, M_comp, p) -> int:
    return int(lib().adaln_bucket_batch(S, M_mem, M_comp, p))


def _host_array(values, ctype):
    arr = (ctype * len(values))(*values)
    return arr, ctypes.cast(arr, ctypes.c_void_p).value


def adaln_bucket_batch_real(S, M_mem, M_comp, p) -> int:
    return int(lib().adaln_bucket_batch_real(S, M_mem, M_comp, float(p)))


def adaln_fit_step_cost(B, S, t, p_lo=1.0, p_hi=3.0, t_budget=0.0) -> dict:
    """Host arrays (sequences) of equal length n; returns a, b, p, rms, M_comp."""
    n = len(t)
    if len(B) != n or len(S) != n:
        raise ValueError("B, S and t must have one length")
    b_arr, b_p = _host_array([int(v) for v in B], ctypes.c_int64)
    s_arr, s_p = _host_array([int(v) for v in S], ctypes.c_int64)
    t_arr, t_p = _host_array([float(v) for v in t], ctypes.c_double)
    out = (ctypes.c_double * 5)()
    _check("adaln_fit_step_cost", lib().adaln_fit_step_cost(
        b_p, s_p, t_p, n, float(p_lo), float(p_hi), float(t_budget), ctypes.cast(out, ctypes.c_void_p)))
    return {"a": out[0], "b": out[1], "p": out[2], "rms": out[3], "M_comp": out[4]}


def adaln_bucket_load_cv(lengths, buckets, M_mem, M_comp, p, rule) -> dict:
    """rule 0: equal-token batches; rule 1: dual constraint. Returns cv, batches, mean."""
    l_arr, l_p = _host_array([int(v) for v in lengths], ctypes.c_int64)
    k_arr, k_p = _host_array([int(v) for v in buckets], ctypes.c_int64)
    out = (ctypes.c_double * 3)()
    _check("adaln_bucket_load_cv", lib().adaln_bucket_load_cv(
        l_p, len(lengths), k_p, len(buckets), M_mem, M_comp, float(p), int(rule),
        ctypes.cast(out, ctypes.c_void_p)))
    return {"cv": out[0], "batches": int(out[1]), "mean": out[2]}


def adaln_status_string(status) -> str:
    return _status_text(status)
