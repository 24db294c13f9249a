"""The pipelined end-to-end step of bench.py (segment chunks on copy-in, compute and
copy-out streams) gives the whole-batch results: y, dx and the statistics bitwise,
dshift/dscale within a summation-order difference."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def test_chunked_end_to_end_step_matches_whole_batch_calls():
    import torch

    import adaln_layernorm_modulate_gb300 as A
    import bench
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(21)
    lens = list(rng.integers(1, 3000, 60))
    w = synth.make("e2e", 21, synth.BF16, 3072, lens, x_mode=synth.ROWS_SCALED, dy_std=0.02)
    dev = torch.device("cuda", 0)

    def host(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)

    h = {k: host(getattr(w, k)) for k in ("x", "dy", "shift", "scale")}
    d = {k: v.to(dev) for k, v in h.items()}
    R, D, nmod, nseg = w.R, w.D, w.nmod, w.nseg
    outs = {"y": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "dx": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
            "mean": torch.empty(R, device=dev), "rstd": torch.empty(R, device=dev),
            "dshift": torch.empty((nmod, D), device=dev), "dscale": torch.empty((nmod, D), device=dev)}
    pin = {k: v.pin_memory() for k, v in h.items()}
    out_h = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in outs.items()}
    chunks = bench.e2e_chunks(w, 6)
    assert chunks is not None and len(chunks) > 2
    sptr = torch.cuda.current_stream().cuda_stream
    step = bench.chunked_e2e_step(A, w, chunks, pin, out_h, d, outs, sptr, lambda: None, dev)
    step()
    step()
    torch.cuda.synchronize()

    cu = torch.from_numpy(w.cu_seqlens.astype(np.int32)).to(dev)
    mod = torch.from_numpy(w.mod_idx.astype(np.int32)).to(dev)
    ref = {k: torch.empty_like(v) for k, v in outs.items()}
    fn = A.adaln_fwd_varlen_workspace_size(R, nseg, D, w.dtype)
    bn = A.adaln_bwd_varlen_workspace_size(R, nseg, nmod, D, w.dtype)
    fws = torch.empty(fn, dtype=torch.uint8, device=dev)
    bws = torch.empty(bn, dtype=torch.uint8, device=dev)
    A.adaln_fwd_varlen(d["x"], d["shift"], d["scale"], ref["y"], ref["mean"], ref["rstd"], cu, mod, nseg,
                       R, nmod, D, bench.EPS, fws, fn, w.dtype, sptr)
    A.adaln_bwd_varlen(d["dy"], d["x"], ref["mean"], ref["rstd"], d["scale"], ref["dx"], ref["dshift"],
                       ref["dscale"], cu, mod, nseg, R, nmod, D, bws, bn, w.dtype, sptr)
    torch.cuda.synchronize()
    for k in ("y", "dx", "mean", "rstd"):
        assert torch.equal(out_h[k], ref[k].cpu()), k
    for k in ("dshift", "dscale"):
        a, b = out_h[k].double(), ref[k].cpu().double()
        assert float((a - b).norm() / b.norm()) < 1e-5, k
