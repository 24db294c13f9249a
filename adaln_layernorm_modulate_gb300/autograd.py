"""Autograd node over libadaln: the fused AdaLN (LayerNorm-Modulate) operator of the
AdaptiveLoad technical summary, section 2.B, as one forward launch and one backward call
(fused dx + D-tile partials, then the fixed-order reduce) in a PyTorch graph.

    y = (x - mean) * rstd * (1 + scale[m]) + shift[m],  rstd = 1 / sqrt(var + eps)

Dense input: x [Bt, N, D], shift and scale [Bt, D]; token (b, n) uses row b.
Packed input: x [R, D] with ``cu_seqlens`` [nseg + 1] and ``mod_idx`` [nseg] (int32, on the
device); segment s uses row ``mod_idx[s]`` of shift and scale [nmod, D].

The node saves x, scale and the fp32 row statistics (8 bytes a row), not y or xhat; with
``save_stats=False`` it keeps no statistics (the forward's are dropped with its outputs) and
the backward recomputes them from x (one more read of x, bitwise the same statistics and
gradients). Every
step runs in the library's kernels; this module only allocates outputs and workspaces
through PyTorch's allocator and passes pointers. dshift and dscale come out of the
library in fp32; autograd wants gradients in the parameters' dtype, so they are rounded
once to it (a no-op for fp32 parameters).
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (ADALN_BF16, ADALN_F32, AdalnError, adaln_bwd, adaln_bwd_recompute,
               adaln_bwd_recompute_workspace_size, adaln_bwd_varlen, adaln_bwd_varlen_recompute,
               adaln_bwd_varlen_recompute_workspace_size, adaln_bwd_varlen_workspace_size,
               adaln_bwd_workspace_size, adaln_fwd, adaln_fwd_varlen, adaln_fwd_varlen_workspace_size,
               adaln_read_status)

__all__ = ["AdaLNModulateFunction", "AdaLNModulate", "adaln_modulate"]


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ADALN_BF16
    if t.dtype == torch.float32:
        return ADALN_F32
    raise TypeError("AdaLN-Modulate supports bfloat16 and float32 tensors, got %s" % t.dtype)


def _workspace(nbytes: int, device) -> torch.Tensor:
    if nbytes <= 0:
        raise AdalnError("workspace size", 2)
    # The caching allocator returns 512-byte aligned blocks; the library needs 256.
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _check_status(ws: torch.Tensor, what: str) -> None:
    st = adaln_read_status(ws)
    if st != 0:
        raise AdalnError(what, st)


class AdaLNModulateFunction(torch.autograd.Function):
    """y = LayerNorm(x) * (1 + scale) + shift with saved fp32 mean/rstd.

    ``check_tables`` reads the packed call's device status after each launch (it
    synchronises the stream): set it while validating new ``cu_seqlens``/``mod_idx``.
    ``save_stats=False``: keep no statistics; the backward recomputes them from x."""

    @staticmethod
    def forward(ctx, x, shift, scale, cu_seqlens=None, mod_idx=None, eps: float = 1e-6,
                check_tables: bool = False, save_stats: bool = True):
        if not x.is_cuda:
            raise ValueError("AdaLN-Modulate runs on CUDA tensors")
        x = x.contiguous()
        shift = shift.contiguous()
        scale = scale.contiguous()
        if shift.dtype != x.dtype or scale.dtype != x.dtype:
            raise TypeError("x, shift and scale must share one dtype")
        dt = _code(x)
        D = x.shape[-1]
        packed = cu_seqlens is not None
        y = torch.empty_like(x)
        if packed:
            if x.dim() != 2 or mod_idx is None:
                raise ValueError("packed input: x [R, D] with cu_seqlens and mod_idx")
            cu = cu_seqlens.to(device=x.device, dtype=torch.int32).contiguous()
            mod = mod_idx.to(device=x.device, dtype=torch.int32).contiguous()
            R, nseg, nmod = x.shape[0], mod.numel(), shift.shape[0]
            mean = torch.empty(R, dtype=torch.float32, device=x.device)
            rstd = torch.empty(R, dtype=torch.float32, device=x.device)
            nb = adaln_fwd_varlen_workspace_size(R, nseg, D, dt)
            ws = _workspace(nb, x.device)
            adaln_fwd_varlen(x, shift, scale, y, mean, rstd, cu, mod, nseg, R, nmod, D, eps, ws, nb, dt)
            if check_tables:
                _check_status(ws, "adaln_fwd_varlen")
            kept = (mean, rstd) if save_stats else (mean[:0], rstd[:0])
            ctx.save_for_backward(x, scale, *kept, cu, mod)
        else:
            if x.dim() != 3 or shift.shape != (x.shape[0], D) or scale.shape != (x.shape[0], D):
                raise ValueError("dense input: x [Bt, N, D], shift and scale [Bt, D]")
            Bt, N = x.shape[0], x.shape[1]
            mean = torch.empty((Bt, N), dtype=torch.float32, device=x.device)
            rstd = torch.empty((Bt, N), dtype=torch.float32, device=x.device)
            adaln_fwd(x, shift, scale, y, mean, rstd, Bt, N, D, eps, dt)
            kept = (mean, rstd) if save_stats else (mean[:0], rstd[:0])
            ctx.save_for_backward(x, scale, *kept)
        ctx.packed = packed
        ctx.check_tables = check_tables
        ctx.save_stats = save_stats
        ctx.eps = eps
        ctx.shift_dtype = shift.dtype
        ctx.mark_non_differentiable(mean, rstd)
        return y, mean, rstd

    @staticmethod
    def backward(ctx, dy, _dmean, _drstd):
        x, scale, mean, rstd = ctx.saved_tensors[:4]
        dy = dy.contiguous()
        dt = _code(x)
        D = x.shape[-1]
        nmod = scale.shape[0]
        dx = torch.empty_like(x)
        dshift = torch.empty((nmod, D), dtype=torch.float32, device=x.device)
        dscale = torch.empty((nmod, D), dtype=torch.float32, device=x.device)
        if ctx.packed:
            cu, mod = ctx.saved_tensors[4:]
            R, nseg = x.shape[0], mod.numel()
            if ctx.save_stats:
                nb = adaln_bwd_varlen_workspace_size(R, nseg, nmod, D, dt)
                ws = _workspace(nb, x.device)
                adaln_bwd_varlen(dy, x, mean, rstd, scale, dx, dshift, dscale, cu, mod, nseg, R, nmod,
                                 D, ws, nb, dt)
            else:
                nb = adaln_bwd_varlen_recompute_workspace_size(R, nseg, nmod, D, dt)
                ws = _workspace(nb, x.device)
                adaln_bwd_varlen_recompute(dy, x, scale, dx, dshift, dscale, cu, mod, nseg, R, nmod, D,
                                           ctx.eps, ws, nb, dt)
            if ctx.check_tables:
                _check_status(ws, "adaln_bwd_varlen")
        else:
            Bt, N = x.shape[0], x.shape[1]
            if ctx.save_stats:
                nb = adaln_bwd_workspace_size(Bt, N, D, dt)
                ws = _workspace(nb, x.device)
                adaln_bwd(dy, x, mean, rstd, scale, dx, dshift, dscale, ws, nb, Bt, N, D, dt)
            else:
                nb = adaln_bwd_recompute_workspace_size(Bt, N, D, dt)
                ws = _workspace(nb, x.device)
                adaln_bwd_recompute(dy, x, scale, dx, dshift, dscale, ws, nb, Bt, N, D, ctx.eps, dt)
        return (dx, dshift.to(ctx.shift_dtype), dscale.to(ctx.shift_dtype), None, None, None, None, None)


def adaln_modulate(x: torch.Tensor, shift: torch.Tensor, scale: torch.Tensor,
                   cu_seqlens: Optional[torch.Tensor] = None, mod_idx: Optional[torch.Tensor] = None,
                   eps: float = 1e-6, check_tables: bool = False, save_stats: bool = True) -> torch.Tensor:
    """Differentiable fused AdaLN-Modulate; returns y (the statistics stay in the graph)."""
    y, _, _ = AdaLNModulateFunction.apply(x, shift, scale, cu_seqlens, mod_idx, eps, check_tables,
                                          save_stats)
    return y


class AdaLNModulate(torch.nn.Module):
    """Module form: ``AdaLNModulate(eps)(x, shift, scale[, cu_seqlens, mod_idx])``. It has no
    parameters of its own: shift and scale come from the conditioning branch."""

    def __init__(self, eps: float = 1e-6, save_stats: bool = True):
        super().__init__()
        self.eps = float(eps)
        self.save_stats = bool(save_stats)

    def forward(self, x, shift, scale, cu_seqlens=None, mod_idx=None):
        return adaln_modulate(x, shift, scale, cu_seqlens, mod_idx, self.eps, save_stats=self.save_stats)

    def extra_repr(self) -> str:
        return "eps=%g, save_stats=%s" % (self.eps, self.save_stats)
