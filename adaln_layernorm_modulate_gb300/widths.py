"""Per-width throughput of the fused forward and backward on the current GPU.

    python -m adaln_layernorm_modulate_gb300.widths [--dims 512,1024,...] [--dtype bf16,f32]
                                                    [--rows N] [--reps N]

For each row width D: one dense batch of random rows (at least 32,760 rows, up to about
512 MB per tensor, or --rows of them), one modulation row; the L2 is flushed by reading a buffer twice its
size before each timed pair of calls; the median of 20 CUDA-event timings of adaln_fwd and
of adaln_bwd (partials and reduce). Prints microseconds and the share of the HBM peak
(algorithmic bytes per call over time; the peak from MEASURED_PEAKS.json when present).
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np
import torch

from . import ADALN_BF16, ADALN_F32, adaln_bwd, adaln_bwd_workspace_size, adaln_fwd

DEFAULT_DIMS = "512,768,1024,1536,2048,2560,3072,4096,5120,6144,8192,10240,12288,14336,16384"


def call_bytes(R: int, D: int, e: int) -> tuple:
    """Each call's own unavoidable traffic, one modulation row."""
    fwd = 2 * R * D * e + 8 * R + 2 * D * e
    bwd = 3 * R * D * e + 8 * R + D * e + 8 * D
    return fwd, bwd


def peak_gbs() -> float:
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


def measure(D: int, dtype: str, dev, flush, fo, reps: int = 20, rows: int = 0) -> tuple:
    code, tdt, e = (ADALN_BF16, torch.bfloat16, 2) if dtype == "bf16" else (ADALN_F32, torch.float32, 4)
    R = rows if rows > 0 else min(262144, max(32760, (512 << 20) // (D * e) // 4 * 4))
    x = torch.randn(R, D, device=dev).to(tdt)
    dy = (0.02 * torch.randn(R, D, device=dev)).to(tdt)
    shift = (0.1 * torch.randn(1, D, device=dev)).to(tdt)
    scale = (0.1 * torch.randn(1, D, device=dev)).to(tdt)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(R, device=dev)
    rstd = torch.empty(R, device=dev)
    dsh = torch.empty(1, D, device=dev)
    dsc = torch.empty(1, D, device=dev)
    nb = adaln_bwd_workspace_size(1, R, D, code)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream

    def fwd():
        adaln_fwd(x, shift, scale, y, mean, rstd, 1, R, D, 1e-6, code, s)

    def bwd():
        adaln_bwd(dy, x, mean, rstd, scale, dx, dsh, dsc, ws, nb, 1, R, D, code, s)

    for _ in range(3):
        fwd()
        bwd()
    marks = []
    for _ in range(reps):
        torch.sum(flush, dim=0, out=fo)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        fwd()
        ev[1].record()
        bwd()
        ev[2].record()
        marks.append(ev)
    torch.cuda.synchronize()
    tf = float(np.median([m[0].elapsed_time(m[1]) for m in marks])) * 1e3
    tb = float(np.median([m[1].elapsed_time(m[2]) for m in marks])) * 1e3
    return R, tf, tb, call_bytes(R, D, e)


def main() -> int:
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--dims", default=DEFAULT_DIMS)
    p.add_argument("--dtype", default="bf16,f32")
    p.add_argument("--rows", type=int, default=0, help="rows a batch (default: by width, as above)")
    p.add_argument("--reps", type=int, default=20, help="timed pairs of calls a width")
    args = p.parse_args()
    dev = torch.device("cuda", torch.cuda.current_device())
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    flush = torch.ones(2 * l2 // 4, device=dev)
    fo = torch.empty((), device=dev)
    peak = peak_gbs()
    print("%-5s %6s %7s | %9s %6s | %9s %6s" % ("dtype", "D", "rows", "fwd us", "peak", "bwd us", "peak"))
    for dtype in args.dtype.split(","):
        for D in (int(v) for v in args.dims.split(",")):
            R, tf, tb, (bf, bb) = measure(D, dtype, dev, flush, fo, args.reps, args.rows)
            print("%-5s %6d %7d | %9.1f %5.1f%% | %9.1f %5.1f%%" % (
                dtype, D, R, tf, 100 * bf / tf / 1e3 / peak, tb, 100 * bb / tb / 1e3 / peak), flush=True)
            torch.cuda.empty_cache()
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
