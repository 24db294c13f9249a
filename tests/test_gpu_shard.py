"""Row sharding on one GPU: adaln_sum_ranks adds stacked per-rank gradients in rank order
(bitwise the float32 rank-order sum), and a batch run as several segment-aligned shards,
each a packed call on its own rows, then summed with adaln_sum_ranks, matches the oracle's
whole-batch results on every row and every modulation row. (Ranks are emulated one after
another on the same device; no kernel waits on another.)"""
import numpy as np
import pytest

import synth
from adaln_layernorm_modulate_gb300 import shard
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import adaln_layernorm_modulate_gb300 as A
    A.lib()


@pytest.mark.parametrize("world,n", [(1, 12), (2, 4096), (3, 6 * 3072), (5, 1001), (8, 2 * 676 * 3072)])
def test_sum_ranks_is_the_rank_order_float32_sum(world, n):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    rng = np.random.default_rng(world * 7919 + n)
    parts = (rng.standard_normal((world, n)) * np.exp(rng.uniform(-20, 20, (world, n)))).astype(np.float32)
    want = parts[0].copy()
    for r in range(1, world):
        want = want + parts[r]
    dp = t.from_numpy(parts).cuda()
    out = t.empty(n, dtype=t.float32, device="cuda")
    A.adaln_sum_ranks(dp, out, world, n)
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_batch_matches_the_oracle(orc, world):
    import adaln_layernorm_modulate_gb300 as A
    t = H.torch()
    w = synth.make("sh", 902, synth.BF16, 3072, [700, 3, 2000, 17, 900, 1, 1500],
                   [2, 0, 1, 2, 0, 3, 1], 4, x_mode=synth.ROWS_SCALED, dy_std=0.02)
    d = H.upload(w)
    y = t.empty((w.R, w.D), dtype=t.bfloat16, device="cuda")
    dx = t.empty_like(y)
    mean = t.empty(w.R, dtype=t.float32, device="cuda")
    rstd = t.empty_like(mean)
    stacked = t.empty((world, 2, w.nmod, w.D), dtype=t.float32, device="cuda")
    for r in range(world):
        sh = shard.make_shard(w.cu_seqlens, w.mod_idx, world, r)
        cu = t.from_numpy(sh.cu_seqlens).cuda()
        mod = t.from_numpy(sh.mod_idx).cuda()
        a, b = sh.row0, sh.row1
        nb = A.adaln_fwd_varlen_workspace_size(sh.rows, sh.nseg, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_fwd_varlen(d.x[a:b], d.shift, d.scale, y[a:b], mean[a:b], rstd[a:b], cu, mod, sh.nseg,
                           sh.rows, w.nmod, w.D, H.EPS, ws, nb, w.dtype)
        assert A.adaln_read_status(ws) == 0
        nb = A.adaln_bwd_varlen_workspace_size(sh.rows, sh.nseg, w.nmod, w.D, w.dtype)
        ws = t.empty(nb, dtype=t.uint8, device="cuda")
        A.adaln_bwd_varlen(d.dy[a:b], d.x[a:b], mean[a:b], rstd[a:b], d.scale, dx[a:b], stacked[r, 0],
                           stacked[r, 1], cu, mod, sh.nseg, sh.rows, w.nmod, w.D, ws, nb, w.dtype)
        assert A.adaln_read_status(ws) == 0
    total = t.empty((2, w.nmod, w.D), dtype=t.float32, device="cuda")
    A.adaln_sum_ranks(stacked, total, world, total.numel())
    t.cuda.synchronize()
    m32, r32 = H.forward_all_rows(orc, w, H.to_host(y, w.dtype), H.to_host(mean, 0), H.to_host(rstd, 0))
    tot = total.cpu().numpy()
    H.backward_all_rows(orc, w, m32, r32, pipeline=(H.to_host(dx, w.dtype), tot[0], tot[1]))
