"""adaln_bwd_noalloc: the dense backward for callers that cannot allocate device memory
(a framework that only lends the tensors it owns, an allocator that must not grow, a plain
C caller). It runs the same kernels with the same launch plan as adaln_bwd, so its dx,
dshift and dscale must be bitwise those of adaln_bwd with a caller workspace, call after
call, while its scratch is the library's own fixed array.

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


def _noalloc(d, mean, rstd, dx, dsh, dsc):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = d.w
    Bt, N = w.dense
    # Straight through the C ABI: no workspace argument exists.
    return A.lib().adaln_bwd_noalloc(d.dy.data_ptr(), d.x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                     d.scale.data_ptr(), dx.data_ptr(), dsh.data_ptr(), dsc.data_ptr(),
                                     Bt, N, w.D, w.dtype, t.cuda.current_stream().cuda_stream)


def _compare(w):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    d = H.upload(w)
    _, mean, rstd, _ = H.gpu_fwd(d)
    dx_ref, dsh_ref, dsc_ref, st = H.gpu_bwd(d, mean, rstd)
    assert st == 0
    dx = t.full_like(dx_ref, float("nan"))
    dsh = t.full_like(dsh_ref, float("nan"))
    dsc = t.full_like(dsc_ref, float("nan"))
    rc = _noalloc(d, mean, rstd, dx, dsh, dsc)
    assert rc == 0, A.adaln_status_string(rc)
    assert A.adaln_noalloc_read_status() == 0
    t.cuda.synchronize()
    assert t.equal(dx, dx_ref), "dx differs from adaln_bwd"
    assert t.equal(dsh, dsh_ref), "dshift differs from adaln_bwd"
    assert t.equal(dsc, dsc_ref), "dscale differs from adaln_bwd"


def test_noalloc_matches_workspace_backward_twice():
    # Three calls in a row with different problems. The first leaves large partials (dy with
    # a standard deviation of 50, 4 samples) all over the scratch; the smaller ones after it
    # must read only what they wrote themselves.
    _compare(synth.dense("na0", 700, synth.F32, 4, 200, 2048, x_mode=synth.ROWS_SCALED, dy_std=50.0))
    _compare(synth.dense("na1", 701, synth.BF16, 2, 1500, 1536, x_mode=synth.ROWS_SCALED, dy_std=0.02))
    _compare(synth.dense("na2", 702, synth.F32, 3, 257, 1024, x_mode=synth.ROWS_SCALED, dy_std=0.02))


def test_noalloc_rejects_problems_beyond_its_scratch():
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    D, Bt, N = 16384, 4, 64
    need = A.adaln_bwd_workspace_size(Bt, N, D, A.ADALN_F32)
    assert need > A.NOALLOC_SCRATCH_BYTES
    # Real buffers of the full problem size: if the size guard ever failed, the kernels
    # would still only touch memory that belongs to the test.
    w = synth.dense("na3", 703, synth.F32, Bt, N, D)
    d = H.upload(w)
    mean = t.zeros(Bt * N, dtype=t.float32, device="cuda")
    rstd = t.ones(Bt * N, dtype=t.float32, device="cuda")
    dx = t.empty((Bt * N, D), dtype=t.float32, device="cuda")
    dsh = t.empty((Bt, D), dtype=t.float32, device="cuda")
    dsc = t.empty((Bt, D), dtype=t.float32, device="cuda")
    rc = _noalloc(d, mean, rstd, dx, dsh, dsc)
    assert A.STATUS[rc] == "ADALN_ERR_WORKSPACE"
    t.cuda.synchronize()


def test_noalloc_status_is_readable():
    """adaln_noalloc_read_status reads the status words a backward leaves at the head of the
    fixed array: after a call they read as OK (the array is zero when the library loads, so
    before the first call on a device there is no status to read)."""
    import adaln_layernorm_modulate_gb300 as A
    before = A.STATUS[A.adaln_noalloc_read_status()]
    assert before in ("ADALN_ERR_WORKSPACE", "ADALN_OK"), before  # OK if a test above ran first
    _compare(synth.dense("na4", 704, synth.BF16, 1, 3000, 1536, x_mode=synth.ROWS_SCALED, dy_std=0.02))
    assert A.adaln_noalloc_read_status() == 0
