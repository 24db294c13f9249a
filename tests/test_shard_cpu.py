"""Row sharding across ranks on CPU: the shard plan, and world-size-2 gloo ranks that each
compute their shard's gradients (here with the oracle) and sum them through
shard.sum_over_ranks. The ordered sum is the exchange step the sharded path adds; these
tests check that every rank gets the same bits, that they equal the local rank-order sum
of the same parts whatever moved them, and that they match the whole batch's gradients."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from adaln_layernorm_modulate_gb300 import shard  # noqa: E402


def test_plan_covers_segments_in_order_and_balances_tokens():
    lens = [256] * 512 + [1024] * 128 + [4096] * 32 + [16384] * 2 + [32760, 75600]
    cu = np.concatenate([[0], np.cumsum(lens)])
    for world in (1, 2, 3, 4, 8, 16):
        plan = shard.plan_shards(cu, world)
        assert len(plan) == world and plan[0][0] == 0 and plan[-1][1] == len(lens)
        assert all(a[1] == b[0] for a, b in zip(plan[:-1], plan[1:]))
        rows = [int(cu[s1] - cu[s0]) for s0, s1 in plan]
        assert sum(rows) == cu[-1]
        # Each cut sits at the first segment boundary at or past the rank's token quantile.
        for r, (s0, s1) in enumerate(plan[:-1]):
            target = -(-int(cu[-1]) * (r + 1) // world)
            assert cu[s1] >= target and (s1 == 0 or cu[s1 - 1] < target or s1 == plan[r][0])


def test_plan_with_few_long_segments_leaves_ranks_empty():
    cu = np.array([0, 100, 300])
    plan = shard.plan_shards(cu, 4)
    assert [p for p in plan if p[1] > p[0]] and sum(p[1] - p[0] for p in plan) == 2
    assert plan[-1][1] == 2


def test_local_tables_start_at_zero_and_keep_modulation_rows():
    cu = np.array([0, 5, 5, 12, 30, 31])
    mod = np.array([3, 0, 3, 1, 2])
    for world in (1, 2, 3):
        got = [shard.make_shard(cu, mod, world, r) for r in range(world)]
        assert sum(s.rows for s in got) == 31
        for s in got:
            assert s.cu_seqlens[0] == 0 and s.cu_seqlens[-1] == s.rows
            assert np.array_equal(s.mod_idx, mod[s.s0:s.s1])
            assert np.array_equal(s.cu_seqlens, cu[s.s0:s.s1 + 1] - cu[s.s0])


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _ordered_sum(stacked, out, world, n):
    acc = stacked[0].numpy().astype(np.float32).copy()
    for r in range(1, world):
        acc = acc + stacked[r].numpy()  # float32 adds, rank order
    out.copy_(__import__("torch").from_numpy(acc))


def _workload():
    return synth.make("shard", 901, synth.F32, 64, [40, 3, 200, 17, 90, 1, 66],
                      [2, 0, 1, 2, 0, 3, 1], 4, x_mode=synth.ROWS_SCALED, dy_std=0.5)


def _shard_grads(w, sh):
    """This shard's fp32 [2, nmod, D] gradients, from the oracle on its rows."""
    import oracle
    orc = oracle.get()
    if sh.rows == 0:
        return np.zeros((2, w.nmod, w.D), np.float32)
    rows = (sh.row0, sh.row1)
    _, mean, rstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod, rows=rows)
    _, dsh, dsc = orc.bwd(w.dy, w.x, mean.astype(np.float32), rstd.astype(np.float32), w.scale, w.dtype,
                          w.cu_seqlens, w.mod_idx, w.nmod, rows=rows)
    return np.stack([dsh, dsc]).astype(np.float32)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = _workload()
    sh = shard.make_shard(w.cu_seqlens, w.mod_idx, world, rank)
    local = torch.from_numpy(_shard_grads(w, sh))
    total = shard.sum_over_ranks(local, reduce=_ordered_sum)
    out.put((rank, total.numpy().tobytes()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_ranks_sum_shard_gradients_in_rank_order(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = _workload()
    # Every rank holds the same bits ...
    assert len(set(got.values())) == 1
    total = np.frombuffer(got[0], dtype=np.float32).reshape(2, w.nmod, w.D)
    # ... which are the local rank-order sum of the shards' parts (the transport adds nothing) ...
    parts = [_shard_grads(w, shard.make_shard(w.cu_seqlens, w.mod_idx, world, r)) for r in range(world)]
    want = parts[0].copy()
    for p in parts[1:]:
        want = want + p
    assert np.array_equal(total, want)
    # ... and the whole batch's gradients to fp32 rounding.
    import oracle
    orc = oracle.get()
    _, mean, rstd = orc.fwd(w.x, w.shift, w.scale, w.dtype, w.cu_seqlens, w.mod_idx, w.nmod)
    _, dsh, dsc = orc.bwd(w.dy, w.x, mean.astype(np.float32), rstd.astype(np.float32), w.scale, w.dtype,
                          w.cu_seqlens, w.mod_idx, w.nmod)
    ref = np.stack([dsh, dsc])
    assert np.linalg.norm(total - ref) <= 1e-6 * np.linalg.norm(ref)
