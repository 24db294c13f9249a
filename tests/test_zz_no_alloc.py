"""adaln_bwd_noalloc: the dense backward for callers that cannot allocate device memory
(a framework that only lends the tensors it owns, an allocator that must not grow, a plain
C caller). It must give what adaln_bwd gives with a caller workspace, call after call,
while its scratch is the library's own fixed array.

This file is collected last on purpose: the entry point's scratch lives for the whole
process, so it runs after every other test has used the library, and it also passes alone
in a fresh process."""
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
    A.lib()


def _compare(w):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    d = H.upload(w)
    Bt, N = w.dense
    _, mean, rstd, _ = H.gpu_fwd(d)
    dx_ref, dsh_ref, dsc_ref, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    dx = t.full_like(dx_ref, float("nan"))
    dsh = t.full_like(dsh_ref, float("nan"))
    dsc = t.full_like(dsc_ref, float("nan"))
    # Straight through the C ABI: no workspace argument exists.
    rc = A.lib().adaln_bwd_noalloc(d.dy.data_ptr(), d.x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                   d.scale.data_ptr(), dx.data_ptr(), dsh.data_ptr(), dsc.data_ptr(),
                                   Bt, N, w.D, w.dtype, t.cuda.current_stream().cuda_stream)
    assert rc == 0, A.adaln_status_string(rc)
    t.cuda.synchronize()
    a, b = H.to_host(dx, w.dtype), H.to_host(dx_ref, w.dtype)
    if w.dtype == synth.BF16:
        diff = np.abs(synth.widen(a, synth.BF16) - synth.widen(b, synth.BF16))
        tol = H.bf16_ulp(b) + 1e-3
    else:
        diff = np.abs(a.astype(np.float64) - b)
        tol = 1e-5 * np.maximum(1.0, np.abs(b.astype(np.float64)))
    assert np.all(diff <= tol), "dx differs from adaln_bwd"
    for got, ref in ((dsh, dsh_ref), (dsc, dsc_ref)):
        assert H.rel_l2(H.to_host(got, 0), H.to_host(ref, 0).astype(np.float64)) <= H.grad_tol(w.dtype)


def test_noalloc_matches_workspace_backward_twice():
    # Two calls in a row with different problems: the second must not see the first's scratch.
    _compare(synth.dense("na1", 701, synth.BF16, 2, 1500, 1536, x_mode=synth.ROWS_SCALED, dy_std=0.02))
    _compare(synth.dense("na2", 702, synth.F32, 3, 257, 1024, x_mode=synth.ROWS_SCALED, dy_std=0.02))


def test_noalloc_rejects_problems_beyond_its_scratch():
    import adaln_layernorm_modulate_gb300 as A
    D, Bt, N = 16384, 4, 64
    need = A.adaln_bwd_workspace_size(Bt, N, D, A.ADALN_F32)
    assert need > A.NOALLOC_SCRATCH_BYTES
    rc = A.lib().adaln_bwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, Bt, N, D, A.ADALN_F32, None)
    assert A.STATUS[rc] == "ADALN_ERR_WORKSPACE"
