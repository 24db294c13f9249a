"""The autograd node over libadaln: it runs the same kernels as the C-ABI calls (bitwise
equal results), its gradients match the oracle, and it refuses CPU tensors."""
import numpy as np
import pytest

import synth
from tests import gpu_harness as H


def test_cpu_tensors_are_refused():
    import torch

    from adaln_layernorm_modulate_gb300.autograd import AdaLNModulate
    m = AdaLNModulate(1e-6)
    assert "eps=1e-06, save_stats=True" in repr(m)
    x = torch.zeros(1, 4, 64)
    with pytest.raises(ValueError):
        m(x, torch.zeros(1, 64), torch.zeros(1, 64))


CASES = {
    "dense-bf16-2x300x1536": lambda: synth.dense("a", 201, synth.BF16, 2, 300, 1536,
                                                 x_mode=synth.ROWS_SCALED, dy_std=0.02),
    "packed-f32-d264": lambda: synth.make("a", 202, synth.F32, 264, [5, 90, 0, 33], [1, 1, 0, 2], 3),
}


@pytest.mark.gpu
@pytest.mark.parametrize("save_stats", [True, False], ids=["saved-stats", "recomputed-stats"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_autograd_matches_direct_calls_and_oracle(orc, name, save_stats):
    import torch

    import adaln_layernorm_modulate_gb300 as A
    from adaln_layernorm_modulate_gb300.autograd import adaln_modulate
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = CASES[name]()
    d = H.upload(w)
    packed = w.dense is None
    x = d.x if packed else d.x.view(w.dense[0], w.dense[1], w.D)
    x = x.clone().requires_grad_(True)
    shift = d.shift.clone().requires_grad_(True)
    scale = d.scale.clone().requires_grad_(True)
    dy = d.dy if packed else d.dy.view(w.dense[0], w.dense[1], w.D)
    if packed:
        y = adaln_modulate(x, shift, scale, d.cu, d.mod, eps=H.EPS, check_tables=True, save_stats=save_stats)
    else:
        y = adaln_modulate(x, shift, scale, eps=H.EPS, save_stats=save_stats)
    y.backward(dy)

    # Same kernels as the C-ABI path: bitwise equal.
    y2, mean2, rstd2, _ = H.gpu_fwd(d)
    dx2, dsh2, dsc2, _ = H.gpu_bwd(d, mean2, rstd2)
    assert torch.equal(y.detach().reshape(w.R, w.D), y2)
    assert torch.equal(x.grad.reshape(w.R, w.D), dx2)
    assert torch.equal(shift.grad, dsh2.to(shift.dtype))
    assert torch.equal(scale.grad, dsc2.to(scale.dtype))

    # And the oracle, within the operator's tolerances.
    ry, rmean, rrstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod, eps=H.EPS)
    H.check_io(H.to_host(y.detach().reshape(w.R, w.D), w.dtype), ry, w.dtype, orc, "y")
    m32, r32 = H.round_f32(rmean), H.round_f32(rrstd)
    rdx, rdsh, rdsc = orc.bwd(w.dy, w.x, m32, r32, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod)
    extra = H.stat_shift_bound(_dx_terms(w, m32, r32))
    H.check_io(H.to_host(x.grad.reshape(w.R, w.D), w.dtype), rdx, w.dtype, orc, "dx", extra=extra)
    tol = H.grad_tol(w.dtype) if w.dtype == synth.F32 else 4e-3  # rounded once to bf16
    assert H.rel_l2(H.to_host(shift.grad.float(), 0), rdsh) <= tol
    assert H.rel_l2(H.to_host(scale.grad.float(), 0), rdsc) <= tol


def _dx_terms(w, mean, rstd):
    x = synth.widen(w.x, w.dtype)
    dy = synth.widen(w.dy, w.dtype)
    m_of_row = np.repeat(w.mod_idx, np.diff(w.cu_seqlens))
    g = dy * (1 + synth.widen(w.scale, w.dtype)[m_of_row])
    xhat = (x - mean[:, None]) * rstd[:, None]
    return rstd, mean, xhat, g.mean(axis=1), (g * xhat).mean(axis=1)
