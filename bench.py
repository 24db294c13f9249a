#!/usr/bin/env python
"""Benchmark of the fused AdaLN hot path on GB300.

One step = one pass of the whole path over one batch: the dual-constraint bucket rule
(host) that shapes the packed batch, the fused forward, the fused backward (dx plus
per-tile D-tile partials) and the fixed-order reduction of dshift/dscale. The default
workload is the packed mixed-length batch at D=3072, bf16 I/O (676 segments, 534,344
tokens); its activations (3.3 GB per tensor) are far larger than L2, so no flush is
needed between steps.

Prints ONE JSON line (rank 0). `value` is algorithmic HBM bytes of forward + backward
divided by the device time of a step (GB/s), over the whole job. Under torchrun every rank
runs an independent replica by default (value summed over ranks, weak scaling); with
`--parallel shard` the ranks split one batch into segment-aligned row shards and each step
ends with the one exchange the path has, the rank-order sum of the modulation gradients
(value = the batch's bytes over the slowest rank's step, strong scaling). `--impl
reference` times the CPU oracle instead, on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "AdaLN fwd+bwd achieved HBM GB/s (% of GB300 peak) and Mtokens/s at D=3072"
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "bwd_partials_traffic.json")
FALLBACK_HBM_GBS = 6800.0
EPS = float(np.float32(1e-6))

WORKLOADS = {
    "packed": 3,          # the headline: packed mixed-length buckets, bf16, D=3072
    "wan-1.3b": 1,
    "wan-14b": 2,
    "mmdit-f32": (4, synth.F32),
    "mmdit-bf16": (4, synth.BF16),
    "bucket-s32760": ("bucket", 32760),  # the packed workload's S=32760 bucket as its own call
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="packed")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--e2e-chunks", type=int, default=8,
                   help="segment chunks of the pipelined end-to-end step (1: serial)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--parallel", choices=["replicas", "shard"], default="replicas",
                   help="under torchrun: every rank runs the whole batch (replicas), or each rank "
                        "runs a segment-aligned row shard and the gradients are summed over ranks "
                        "in rank order (shard)")
    p.add_argument("--max-tokens", type=int, default=0,
                   help="keep only the leading segments holding at most this many tokens "
                        "(a smaller case of the same workload, e.g. for profiler captures)")
    return p.parse_args()


# ------------------------------------------------------------------------------------------
# workload and byte accounting
# ------------------------------------------------------------------------------------------
def make_workload(name: str, bucket_batch=None, generate=True, max_tokens=0) -> synth.Workload:
    spec = WORKLOADS[name]
    if spec == 3 or (isinstance(spec, tuple) and spec[0] == "bucket"):
        if bucket_batch is None:
            import oracle
            bucket_batch = oracle.bucket_batch
        if spec == 3:
            w = synth.config(3, bucket_batch=bucket_batch, generate=False)
        else:
            w = synth.bucket(spec[1], bucket_batch, generate=False)
    elif isinstance(spec, tuple):
        w = synth.config(spec[0], dtype=spec[1], generate=False)
    else:
        w = synth.config(spec, generate=False)
    if max_tokens and w.R > max_tokens:
        keep = int(np.searchsorted(w.cu_seqlens, max_tokens, side="right")) - 1
        if keep < 1:
            raise ValueError("--max-tokens keeps no segment")
        w.cu_seqlens = w.cu_seqlens[:keep + 1].copy()
        w.mod_idx = w.mod_idx[:keep].copy()
        w.nmod = int(w.mod_idx.max()) + 1
        w.name += "-first%dtok" % w.R
        if w.dense is not None:
            w.dense = (keep, w.dense[1])
        w.meta.pop("batches", None)
        w.meta.pop("bucket_s", None)
    if generate:
        synth.fill(w)
    return w


def describe(w: synth.Workload) -> dict:
    return {
        "workload": w.name,
        "tokens": w.R, "D": w.D, "segments": w.nseg, "modulation_rows": w.nmod,
        "layout": "dense [Bt,N,D]" if w.dense else "packed cu_seqlens",
        "io_dtype": synth.DTYPE_NAMES[w.dtype], "stats_and_grads": "f32",
        "parallelism": "replicas",
    }


def algorithmic_bytes(R: int, D: int, e: int, nmod: int) -> dict:
    """Minimum HBM traffic of each call: every tensor it must read or write, once."""
    fwd = R * D * e + R * D * e + 8 * R + 2 * nmod * D * e          # x, y, mean+rstd, shift+scale
    partials = 2 * R * D * e + 8 * R + R * D * e + nmod * D * e      # dy, x, stats, dx, scale
    reduce = 8 * nmod * D                                            # dshift, dscale
    return {"fwd": fwd, "bwd_partials": partials, "bwd_reduce": reduce, "bwd": partials + reduce,
            "step": fwd + partials + reduce}


def literal_bytes(R: int, D: int, e: int, nmod: int) -> int:
    """Each tensor of the pass counted once: read x, dy and the modulation tables, write y,
    dx, the statistics and the gradients. The calls' own traffic also reads x a second time
    and the statistics back (in the backward): 1.25x this on the row tensors."""
    return 4 * R * D * e + 8 * R + 2 * nmod * D * e + 8 * nmod * D


def hbm_peak():
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha() -> str:
    """Hash of the backward kernel's code (its sources with comments and blank space
    removed): a recorded traffic figure stays valid across comment edits, not code edits."""
    h = hashlib.sha256()
    for rel in ("adaln_layernorm_modulate_gb300/csrc/bwd.cu", "adaln_layernorm_modulate_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the backward partials kernel from the committed ncu summary,
    or None if it was taken on another workload or before the kernel last changed."""
    try:
        with open(TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("source_sha256") != kernel_sources_sha():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            import torch
            ident = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            ident = str(device_index)
        self.ident = ident

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for name, flag in zip(self.NAMES, parts[4:8]):
                    if flag.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------
# distributed plumbing (replicas: barrier + max only)
# ------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend="gloo"):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ------------------------------------------------------------------------------------------
def oracle_rows_time(orc, w: synth.Workload, r0: int, r1: int) -> float:
    t0 = time.perf_counter()
    _, mean, rstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod, eps=EPS,
                            rows=(r0, r1))
    orc.bwd(w.dy, w.x, mean.astype(np.float32), rstd.astype(np.float32), w.scale, w.dtype,
            w.cu_seqlens, w.mod_idx, w.nmod, rows=(r0, r1))
    return time.perf_counter() - t0


def sample_bytes(w: synth.Workload, rows: int) -> int:
    e = 2 if w.dtype == synth.BF16 else 4
    b = algorithmic_bytes(rows, w.D, e, 0)
    return b["fwd"] + b["bwd_partials"]


def cpu_baseline(w: synth.Workload, seconds: float) -> dict:
    """The oracle timed on the host: on all cores (row blocks on one thread per core, the
    reported value) and on one thread, each on a sample of the workload's leading tokens sized
    to about `seconds` of wall time."""
    import oracle
    orc = oracle.get()
    cores = os.cpu_count() or 1
    calib = min(w.R, 2048)
    per_row = oracle_rows_time(orc, w, 0, calib) / calib
    rows1 = int(min(w.R, max(64, seconds / max(per_row, 1e-9))))
    dt1 = oracle_rows_time(orc, w, 0, rows1)
    rowsn = int(min(w.R, max(64, seconds * cores / max(per_row, 1e-9))))
    t0 = time.perf_counter()
    orc.fwd_bwd_blocks(w.x, w.dy, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod,
                       (0, rowsn), cores, eps=EPS)
    dtn = time.perf_counter() - t0
    return {"value": sample_bytes(w, rowsn) / dtn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "forward + backward of the first %d of %d tokens in blocks of 1024 rows on %d "
                      "threads (%.1f s, fp64)" % (rowsn, w.R, cores, dtn),
            "mtokens_per_s": rowsn / dtn / 1e6,
            "single_thread": {"value": sample_bytes(w, rows1) / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": "forward + backward of the first %d tokens (%.1f s)" % (rows1, dt1),
                              "mtokens_per_s": rows1 / dt1 / 1e6}}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on all of the host's cores (row blocks
    on one thread per core), each step a bounded sample of the workload (consecutive tokens
    at a seeded offset) sized so that the whole run takes about 90 s."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = make_workload(args.workload, max_tokens=args.max_tokens)
    orc = oracle.get()
    cores = os.cpu_count() or 1
    per_row = oracle_rows_time(orc, w, 0, 64) / 64
    total_steps = args.steps + args.warmup
    rows = int(max(16, min(w.R, 90.0 / total_steps * cores / max(per_row, 1e-9))))
    starts = np.random.default_rng(0).integers(0, max(1, w.R - rows), total_steps)

    def one(i):
        t0 = time.perf_counter()
        orc.fwd_bwd_blocks(w.x, w.dy, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod,
                           (int(starts[i]), int(starts[i]) + rows), cores, eps=EPS)
        return time.perf_counter() - t0

    for i in range(args.warmup):
        one(i)
    t = sum(one(i) for i in range(args.warmup, total_steps))
    ms = t / args.steps * 1e3
    gbs = sample_bytes(w, rows) / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: forward + backward of %d consecutive tokens at a seeded "
                                   "offset of the %d-token workload, in blocks of 1024 rows on %d "
                                   "threads (fp64)" % (rows, w.R, cores)},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "mtokens_per_s": rows / (ms / 1e3) / 1e6,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------
def e2e_chunks(w: synth.Workload, n: int):
    """Split a packed batch into about n chunks of consecutive segments for the end-to-end
    pipeline, or None if the chunks' modulation rows would not be contiguous, disjoint and
    covering (every table row must be written by exactly one chunk's backward)."""
    if w.dense is not None or w.nseg < 2:
        return None
    mod = np.asarray(w.mod_idx)
    if w.nmod != w.nseg or not np.array_equal(mod, np.arange(w.nseg)):
        return None
    cu = np.asarray(w.cu_seqlens)
    cuts = sorted(set(int(np.searchsorted(cu, w.R * i / n)) for i in range(1, n)) - {0, w.nseg})
    bounds = [0] + cuts + [w.nseg]
    return [(s0, s1) for s0, s1 in zip(bounds[:-1], bounds[1:]) if s1 > s0]


def chunked_e2e_step(A, w, chunks, pin, out_h, d, outs, sptr, shape_batch, dev):
    """One end-to-end step over segment chunks: chunk c's inputs go up on a copy stream, its
    forward and backward run on the compute stream once they have landed, and its outputs
    come down on a third stream, so copies in both directions overlap the kernels and each
    other. Each chunk is a packed call on its own segments and table rows. Consecutive steps
    alternate between two sets of device buffers (inputs, tables, outputs), so a step's
    inputs go up while the step before it is still computing and copying its results down;
    a set is refilled only once the step that last used it has read its inputs and copied
    its outputs down. `step.finish()` makes the compute stream wait for every copy issued."""
    import torch
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cu = np.asarray(w.cu_seqlens)
    rows = ("x", "dy")
    tables = ("shift", "scale")
    out_rows = ("y", "dx", "mean", "rstd")
    out_tables = ("dshift", "dscale")
    host_tables = []
    ws_f = ws_b = 0
    for s0, s1 in chunks:
        t0, t1 = int(cu[s0]), int(cu[s1])
        host_tables.append((torch.from_numpy((cu[s0:s1 + 1] - t0).astype(np.int32)).pin_memory(),
                            torch.from_numpy(np.arange(s1 - s0, dtype=np.int32)).pin_memory()))
        R, nseg = t1 - t0, s1 - s0
        ws_f = max(ws_f, A.adaln_fwd_varlen_workspace_size(R, nseg, w.D, w.dtype))
        ws_b = max(ws_b, A.adaln_bwd_varlen_workspace_size(R, nseg, nseg, w.D, w.dtype))
    wsf = torch.empty(ws_f, dtype=torch.uint8, device=dev)  # compute-stream order: one suffices
    wsb = torch.empty(ws_b, dtype=torch.uint8, device=dev)

    def buffer_set(dd, oo):
        tabs = [(torch.empty(hc.numel(), dtype=torch.int32, device=dev),
                 torch.empty(hm.numel(), dtype=torch.int32, device=dev)) for hc, hm in host_tables]
        return {"d": dd, "o": oo, "tables": tabs, "read": None, "written": None}

    sets = [buffer_set(d, outs),
            buffer_set({k: torch.empty_like(d[k]) for k in rows + tables},
                       {k: torch.empty_like(v) for k, v in outs.items()})]
    state = {"k": 0}

    def step():
        shape_batch()
        bs = sets[state["k"] % 2]
        state["k"] += 1
        if bs["read"] is not None:
            s_in.wait_event(bs["read"])      # this set's inputs are no longer read
            comp.wait_event(bs["written"])   # its outputs have been copied down
        dd, oo = bs["d"], bs["o"]
        for (s0, s1), (hcu, hmod), (dcu, dmod) in zip(chunks, host_tables, bs["tables"]):
            t0, t1 = int(cu[s0]), int(cu[s1])
            with torch.cuda.stream(s_in):
                for k in rows:
                    dd[k][t0:t1].copy_(pin[k][t0:t1], non_blocking=True)
                for k in tables:
                    dd[k][s0:s1].copy_(pin[k][s0:s1], non_blocking=True)
                dcu.copy_(hcu, non_blocking=True)
                dmod.copy_(hmod, non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_in)
            comp.wait_event(landed)
            R, nseg = t1 - t0, s1 - s0
            A.adaln_fwd_varlen(dd["x"][t0:t1], dd["shift"][s0:s1], dd["scale"][s0:s1], oo["y"][t0:t1],
                               oo["mean"][t0:t1], oo["rstd"][t0:t1], dcu, dmod, nseg, R, nseg, w.D,
                               EPS, wsf, ws_f, w.dtype, sptr)
            A.adaln_bwd_varlen(dd["dy"][t0:t1], dd["x"][t0:t1], oo["mean"][t0:t1], oo["rstd"][t0:t1],
                               dd["scale"][s0:s1], oo["dx"][t0:t1], oo["dshift"][s0:s1],
                               oo["dscale"][s0:s1], dcu, dmod, nseg, R, nseg, w.D, wsb, ws_b,
                               w.dtype, sptr)
            done = torch.cuda.Event()
            done.record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for k in out_rows:
                    out_h[k][t0:t1].copy_(oo[k][t0:t1], non_blocking=True)
                for k in out_tables:
                    out_h[k][s0:s1].copy_(oo[k][s0:s1], non_blocking=True)
        bs["read"] = torch.cuda.Event()
        bs["read"].record(comp)
        bs["written"] = torch.cuda.Event()
        bs["written"].record(s_out)

    def finish():
        for bs in sets:
            if bs["written"] is not None:
                comp.wait_event(bs["written"])

    step.finish = finish
    step.h2d_bytes = sum(pin[k].element_size() * pin[k].numel() for k in rows + tables) + sum(
        (hc.numel() + hm.numel()) * 4 for hc, hm in host_tables)
    return step


def run_ours(args):
    import torch

    import adaln_layernorm_modulate_gb300 as A

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    # The sharded path's gradient exchange moves device tensors (NCCL); replicas only need a
    # barrier and a max of times.
    dist = dist_init(world, "nccl" if args.parallel == "shard" else "gloo")
    dev = torch.device("cuda", local)

    w = make_workload(args.workload, bucket_batch=A.adaln_bucket_batch, max_tokens=args.max_tokens)
    full = w
    sharded = args.parallel == "shard"
    if sharded:
        # This rank's rows: a segment-aligned shard of the batch, as a packed call on its own
        # segments with the batch's modulation tables.
        from adaln_layernorm_modulate_gb300 import shard as S
        sh = S.make_shard(w.cu_seqlens, w.mod_idx, world, rank)
        w = synth.Workload(name=w.name, seed=w.seed, dtype=w.dtype, D=w.D,
                           cu_seqlens=sh.cu_seqlens.astype(np.int64), mod_idx=sh.mod_idx.astype(np.int64),
                           nmod=w.nmod, dense=None, x=w.x[sh.row0:sh.row1], dy=w.dy[sh.row0:sh.row1],
                           shift=w.shift, scale=w.scale, meta=dict(w.meta))
    e = 2 if w.dtype == synth.BF16 else 4
    tdt = torch.bfloat16 if w.dtype == synth.BF16 else torch.float32
    packed = w.dense is None

    def host_tensor(a):
        if w.dtype == synth.BF16 and a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(a)

    h = {k: host_tensor(getattr(w, k)) for k in ("x", "dy", "shift", "scale")}
    h["cu"] = torch.from_numpy(w.cu_seqlens.astype(np.int32))
    h["mod"] = torch.from_numpy(w.mod_idx.astype(np.int32))
    d = {k: v.to(dev) for k, v in h.items()}
    R, D, nmod, nseg = w.R, w.D, w.nmod, w.nseg
    y = torch.empty((R, D), dtype=tdt, device=dev)
    dx = torch.empty((R, D), dtype=tdt, device=dev)
    mean = torch.empty(R, dtype=torch.float32, device=dev)
    rstd = torch.empty(R, dtype=torch.float32, device=dev)
    grads = torch.empty((2, nmod, D), dtype=torch.float32, device=dev)
    dshift, dscale = grads[0], grads[1]
    if packed:
        fws_n = A.adaln_fwd_varlen_workspace_size(R, nseg, D, w.dtype)
        bws_n = A.adaln_bwd_varlen_workspace_size(R, nseg, nmod, D, w.dtype)
    else:
        fws_n = 0
        bws_n = A.adaln_bwd_workspace_size(w.dense[0], w.dense[1], D, w.dtype)
    fws = torch.empty(max(fws_n, 1), dtype=torch.uint8, device=dev)
    bws = torch.empty(bws_n, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    buckets = w.meta.get("batches")

    def shape_batch():
        # Row a1 of the path: the bucket rule that sized this packed batch (host integers).
        if buckets is not None:
            got = [A.adaln_bucket_batch(S, synth.BUCKET_M_MEM, synth.BUCKET_M_COMP, synth.BUCKET_P)
                   for S in w.meta["bucket_s"]]
            if got != buckets:
                raise RuntimeError("bucket sizes changed")

    def fwd(x, shift, scale, cu, mod):
        if packed:
            A.adaln_fwd_varlen(x, shift, scale, y, mean, rstd, cu, mod, nseg, R, nmod, D, EPS, fws,
                               fws_n, w.dtype, sptr)
        else:
            A.adaln_fwd(x, shift, scale, y, mean, rstd, w.dense[0], w.dense[1], D, EPS, w.dtype, sptr)

    def bwd_stage(stage, dy, x, scale, cu, mod):
        if packed:
            fn = {"partials": A.adaln_bwd_varlen_partials, "reduce": A.adaln_bwd_varlen_reduce,
                  "both": A.adaln_bwd_varlen}[stage]
            fn(dy, x, mean, rstd, scale, dx, dshift, dscale, cu, mod, nseg, R, nmod, D, bws, bws_n,
               w.dtype, sptr)
        else:
            fn = {"partials": A.adaln_bwd_partials, "reduce": A.adaln_bwd_reduce,
                  "both": A.adaln_bwd}[stage]
            fn(dy, x, mean, rstd, scale, dx, dshift, dscale, bws, bws_n, w.dense[0], w.dense[1], D,
               w.dtype, sptr)

    def step(ev):
        # ev: None (no events), [begin, end], [begin, after fwd, after partials, end], or, when
        # each timed call gets its own L2 flush, [begin, after fwd, after the flush, after
        # partials, end]. An event recorded between two launches costs about 2 us of GPU time
        # on GB300, so the headline steps record none between their calls; a second pass times
        # each call.
        shape_batch()
        if ev:
            ev[0].record(stream)
        fwd(d["x"], d["shift"], d["scale"], d["cu"], d["mod"])
        if ev and len(ev) >= 4:
            ev[1].record(stream)
        if ev and len(ev) == 5:
            torch.sum(flush, dim=0, out=flush_sum)
            ev[2].record(stream)
        bwd_stage("partials", d["dy"], d["x"], d["scale"], d["cu"], d["mod"])
        if ev and len(ev) >= 4:
            ev[-2].record(stream)
        bwd_stage("reduce", d["dy"], d["x"], d["scale"], d["cu"], d["mod"])
        if sharded and dist is not None:
            # The one exchange of the sharded path: every rank's gradients, gathered and
            # summed in rank order (adaln_sum_ranks), the same bits on every rank.
            S.sum_over_ranks(grads)
        if ev:
            ev[-1].record(stream)

    def events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    for _ in range(args.warmup):
        step(events(4))
    if packed:
        st = A.adaln_read_status(bws, sptr)
        if st != 0:
            raise RuntimeError("device status %s" % A.adaln_status_string(st))
    torch.cuda.synchronize()

    # A step whose activations could stay in L2 (129 MB on GB300) from the step before
    # is preceded by a read of a buffer twice the L2 size: it evicts the previous step's
    # lines (writing back the dirty ones) and leaves only clean lines behind, so the step
    # neither hits in L2 nor pays for someone else's write-backs. The flush falls outside
    # the step's events, and the step time is then the sum of its calls.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    tensor_bytes = R * D * e
    flush = None
    if tensor_bytes < 2 * l2_bytes:
        flush = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        flush_sum = torch.empty((), dtype=torch.float32, device=dev)
        l2_note = "L2 flushed before each step (%.0f MB read, outside the timed calls)" % (flush.numel() * 4 / 1e6)
    else:
        l2_note = "activations larger than L2 (%.2f GB per tensor); no flush" % (tensor_bytes / 1e9)

    def run_steps(per_step, flushed=True):
        # K steps, each preceded by the L2 flush when there is one (outside its events).
        step_events = [per_step() for _ in range(args.steps)]
        t0, t1 = events(2)
        barrier(dist)
        torch.cuda.synchronize()
        t0.record(stream)
        for ev in step_events:
            if flush is not None and flushed:
                torch.sum(flush, dim=0, out=flush_sum)
            step(ev)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        return t0, t1, step_events

    clocks = ClockSampler(local)
    clocks.start()
    # The timed steps: events only around each step (none at all without a flush).
    t0, t1, step_events = run_steps(lambda: events(2) if flush is not None else None)
    if flush is None:
        step_ms = t0.elapsed_time(t1) / args.steps
    else:
        step_ms = float(np.mean([ev[0].elapsed_time(ev[1]) for ev in step_events]))
    ms_per_step = max_over_ranks(dist, step_ms)
    # The per-call breakdown (and the roofline's kernel time): the same K steps again with
    # events between the calls. Where the activations fit in L2 the backward also gets its
    # own flush (a read, outside its events), as each timed call does: otherwise the
    # forward's output, still dirty in L2, would be written back inside the backward's time.
    _, _, split = run_steps(lambda: events(5 if flush is not None else 4))
    # Where the steps are flushed, also the steady back-to-back rate without the flush (each
    # step then also writes back the previous step's outputs left dirty in L2): a secondary
    # figure.
    steady = None
    if flush is not None:
        s0, s1, _ = run_steps(lambda: None, flushed=False)
        steady_ms = max_over_ranks(dist, s0.elapsed_time(s1) / args.steps)
    clk = clocks.stop()
    fwd_ms = float(np.mean([ev[0].elapsed_time(ev[1]) for ev in split]))
    part_ms = float(np.mean([ev[-3].elapsed_time(ev[-2]) for ev in split]))
    red_ms = float(np.mean([ev[-2].elapsed_time(ev[-1]) for ev in split]))

    nb = algorithmic_bytes(R, D, e, nmod)
    # Whole-job bytes: every replica's batch, or the one batch the shards split.
    job_bytes = algorithmic_bytes(full.R, D, e, nmod)["step"] if sharded else world * nb["step"]
    value = job_bytes / (ms_per_step / 1e3) / 1e9
    if flush is not None:
        steady = {"note": "back-to-back steps without the L2 flush: each step also writes back the "
                          "previous step's outputs still dirty in L2, which the flushed figure above "
                          "leaves to the flush outside its timed region",
                  "ms_per_step": steady_ms, "value": job_bytes / (steady_ms / 1e3) / 1e9, "unit": "GB/s"}
    peak, peak_src = hbm_peak()
    if steady is not None:
        steady["pct_of_peak"] = 100.0 * steady["value"] / (world * peak)

    # End to end through the public calls, host buffers in and out, copies inside the region.
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        pin = {k: v.pin_memory() for k, v in h.items()}
        out_h = {"y": torch.empty_like(y, device="cpu").pin_memory(),
                 "dx": torch.empty_like(dx, device="cpu").pin_memory(),
                 "mean": torch.empty_like(mean, device="cpu").pin_memory(),
                 "rstd": torch.empty_like(rstd, device="cpu").pin_memory(),
                 "dshift": torch.empty_like(dshift, device="cpu").pin_memory(),
                 "dscale": torch.empty_like(dscale, device="cpu").pin_memory()}
        outs = {"y": y, "dx": dx, "mean": mean, "rstd": rstd, "dshift": dshift, "dscale": dscale}
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(v.numel() * v.element_size() for v in out_h.values())

        def e2e_step():
            for k, v in pin.items():
                d[k].copy_(v, non_blocking=True)
            shape_batch()
            fwd(d["x"], d["shift"], d["scale"], d["cu"], d["mod"])
            bwd_stage("both", d["dy"], d["x"], d["scale"], d["cu"], d["mod"])
            for k, v in out_h.items():
                v.copy_(outs[k], non_blocking=True)

        chunks = e2e_chunks(w, args.e2e_chunks) if args.e2e_chunks > 1 else None
        if chunks is not None:
            e2e_step = chunked_e2e_step(A, w, chunks, pin, out_h, d, outs, sptr, shape_batch, dev)
            h2d = e2e_step.h2d_bytes
        e2e_step()
        if chunks is not None:
            e2e_step()  # both buffer sets warmed up
            e2e_step.finish()
        torch.cuda.synchronize()
        a, b = events(2)
        barrier(dist)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        if chunks is not None:
            e2e_step.finish()  # the region ends when the last copy has landed
        b.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        e2e_ms = max_over_ranks(dist, a.elapsed_time(b) / args.e2e_steps)
        e2e = {"value": job_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipeline": ("%d segment chunks; host-to-device copies, kernels and device-to-host "
                            "copies on three streams, two buffer sets alternating between steps"
                            % len(chunks)) if chunks else "serial"}

    if rank != 0:
        return 0
    base = None if args.no_cpu_baseline or world > 1 else cpu_baseline(w, args.cpu_seconds)
    achieved = nb["bwd_partials"] / (part_ms / 1e3) / 1e9
    traffic = recorded_traffic(w.name)
    lit = world * literal_bytes(R, D, e, nmod)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if sharded else "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": dict(describe(full), parallelism=("row shards (segment-aligned), gradients summed "
                                                    "over ranks in rank order" if sharded else "replicas")),
        "l2": l2_note,
        "pct_of_peak": 100.0 * value / (world * peak),
        "mtokens_per_s": (full.R if sharded else world * R) / (ms_per_step / 1e3) / 1e6,
        "steady_no_flush": steady,
        "literal_bytes": {
            "note": "each tensor of the pass counted once (read x, dy, shift, scale; write y, dx, "
                    "mean, rstd, dshift, dscale); value above counts each call's own traffic",
            "bytes_per_step": lit, "value": lit / (ms_per_step / 1e3) / 1e9, "unit": "GB/s",
            "pct_of_peak": 100.0 * lit / (ms_per_step / 1e3) / 1e9 / (world * peak)},
        "per_call_us": {"fwd": fwd_ms * 1e3, "bwd_partials": part_ms * 1e3, "bwd_reduce": red_ms * 1e3,
                        "bwd": (part_ms + red_ms) * 1e3},
        "per_call_gbs": {"fwd": nb["fwd"] / fwd_ms / 1e6, "bwd": nb["bwd"] / (part_ms + red_ms) / 1e6},
        "algorithmic_bytes_per_step": nb["step"],
        "roofline": {"kernel": "bwd_kernel (fused dx + D-tile partials)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_source": peak_src + " hbm_gbs",
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if traffic is None else float(traffic),
                     "algorithmic_bytes": nb["bwd_partials"]},
        "cpu_baseline": base,
        "e2e": e2e,
        "gpu_launches": (4 if sharded and world > 1 else 3) * args.steps,
        "per_call_note": ("per_call_us and roofline.achieved come from a second pass of the same %d "
                          "steps with CUDA events between the calls%s; the timed steps record none "
                          "there (each such event costs ~2 us of GPU time)"
                          % (args.steps, ", and an L2 flush before the backward as before the forward"
                             if flush is not None else "")),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
