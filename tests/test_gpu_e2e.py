"""The pipelined end-to-end step of bench.py (segment chunks on copy-in, compute and
copy-out streams, two device buffer sets alternating between steps) gives bitwise the results of the same chunk calls made one after another
on one stream (so no copy overtakes a launch that needs it), and the whole-batch call's
results within rounding: a chunk's forward may map its rows differently from the whole
batch's (tile length decides between the two forward stagings for some bf16 widths), which
changes the summation order of the row statistics."""
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
    for _ in range(3):  # both buffer sets, then the first one refilled
        step()
    step.finish()
    torch.cuda.synchronize()

    cu = np.asarray(w.cu_seqlens)
    ref = {k: torch.empty_like(v) for k, v in outs.items()}
    for s0, s1 in chunks:
        t0, t1 = int(cu[s0]), int(cu[s1])
        r, ns = t1 - t0, s1 - s0
        lcu = torch.from_numpy((cu[s0:s1 + 1] - t0).astype(np.int32)).to(dev)
        lmod = torch.arange(ns, dtype=torch.int32, device=dev)
        fn = A.adaln_fwd_varlen_workspace_size(r, ns, w.D, w.dtype)
        bn = A.adaln_bwd_varlen_workspace_size(r, ns, ns, w.D, w.dtype)
        fws = torch.empty(fn, dtype=torch.uint8, device=dev)
        bws = torch.empty(bn, dtype=torch.uint8, device=dev)
        A.adaln_fwd_varlen(d["x"][t0:t1], d["shift"][s0:s1], d["scale"][s0:s1], ref["y"][t0:t1],
                           ref["mean"][t0:t1], ref["rstd"][t0:t1], lcu, lmod, ns, r, ns, D, bench.EPS,
                           fws, fn, w.dtype, sptr)
        A.adaln_bwd_varlen(d["dy"][t0:t1], d["x"][t0:t1], ref["mean"][t0:t1], ref["rstd"][t0:t1],
                           d["scale"][s0:s1], ref["dx"][t0:t1], ref["dshift"][s0:s1], ref["dscale"][s0:s1],
                           lcu, lmod, ns, r, ns, D, bws, bn, w.dtype, sptr)
    torch.cuda.synchronize()
    for k in outs:
        assert torch.equal(out_h[k], ref[k].cpu()), k

    # The whole batch in one call.
    dcu = torch.from_numpy(w.cu_seqlens.astype(np.int32)).to(dev)
    dmod = torch.from_numpy(w.mod_idx.astype(np.int32)).to(dev)
    whole = {k: torch.empty_like(v) for k, v in outs.items()}
    fn = A.adaln_fwd_varlen_workspace_size(R, nseg, D, w.dtype)
    bn = A.adaln_bwd_varlen_workspace_size(R, nseg, nmod, D, w.dtype)
    fws = torch.empty(fn, dtype=torch.uint8, device=dev)
    bws = torch.empty(bn, dtype=torch.uint8, device=dev)
    A.adaln_fwd_varlen(d["x"], d["shift"], d["scale"], whole["y"], whole["mean"], whole["rstd"], dcu, dmod,
                       nseg, R, nmod, D, bench.EPS, fws, fn, w.dtype, sptr)
    A.adaln_bwd_varlen(d["dy"], d["x"], whole["mean"], whole["rstd"], d["scale"], whole["dx"],
                       whole["dshift"], whole["dscale"], dcu, dmod, nseg, R, nmod, D, bws, bn,
                       w.dtype, sptr)
    torch.cuda.synchronize()
    for k in ("mean", "rstd"):
        a, b = out_h[k].double(), whole[k].cpu().double()
        assert float((a - b).abs().max() / b.abs().max()) < 1e-5, k
    for k, tol in (("y", 4e-3), ("dx", 4e-3), ("dshift", 1e-4), ("dscale", 1e-4)):
        a, b = out_h[k].double(), whole[k].cpu().double()
        assert float((a - b).norm() / b.norm()) < tol, k
