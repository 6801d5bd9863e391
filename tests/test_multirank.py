"""The multi-rank host logic of bench.py on two gloo ranks (CPU): every rank
gets its own seeded batch of the same shape, the work is the same per rank
(weak scaling), and the step time is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import synth

    cfg = bench.rank_config(synth.C1.replace(hq=2, hk=2, s=256), rank)
    x = synth.prefill(cfg)
    r = oracle.sparge_block_map(x["q"], x["k"], synth.per_head(cfg, 0.5), None,
                                synth.per_head(cfg, cfg.simthreshd1), cfg.scale, False, False,
                                dtype="f16")
    tiles = torch.tensor([int(r["count"].sum())], dtype=torch.int64)
    gathered = [torch.zeros_like(tiles) for _ in range(world)]
    dist.all_gather(gathered, tiles)
    slowest = bench.max_over_ranks(1.0 + rank, world)
    np.save(os.path.join(out_dir, f"r{rank}.npy"),
            np.array([cfg.seed, int(x["q"].astype(np.int64).sum()), slowest] +
                     [int(g.item()) for g in gathered]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = (np.load(tmp_path / f"r{r}.npy") for r in range(world))
    import synth
    import bench

    assert r0[0] == synth.C1.seed and r1[0] != r0[0]          # own batch per rank
    assert r0[1] != r1[1]                                      # different data
    assert r0[2] == 2.0 and r1[2] == 2.0                       # max over ranks
    assert (r0[3:] == r1[3:]).all()                            # same gathered view
    assert r0[3] == r0[3 + 0] and r0[3] > 0 and r0[4] > 0      # work on both ranks
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _cp_worker(rank, world, port, out_dir):
    """One context-parallel rank on CPU: the oracle stands in for the GPU
    partial of this rank's kv range; the exchange is the library's own
    all-gather."""
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from fmha_block_map_gb300 import cp

    rng = np.random.default_rng(7)
    q = rng.standard_normal((256, 32))
    k = rng.standard_normal((1000, 32))
    v = rng.standard_normal((1000, 16))
    rows = {2: [0, 3, 8, 9, 15], 3: [1, 2, 14]}           # q block -> LUT row
    lo, hi = cp.kv_shard_bounds(16, world)[rank]
    r0, r1 = cp.shard_rows(1000, lo, hi)
    o = np.zeros((2, 64, 16))
    l = np.zeros((2, 64))
    for n, (i, row) in enumerate(sorted(rows.items())):
        sub = oracle.shard_lut_row(row, lo, hi)
        o[n], l[n] = oracle.attention_unit(q, k[r0:r1], v[r0:r1], sub, i, 64, 64, 0.3, False)
    o_all, l_all = cp.gather_partials(torch.from_numpy(o), torch.from_numpy(l))
    res = []
    for n, (i, row) in enumerate(sorted(rows.items())):
        got = oracle.combine(o_all[:, n].numpy(), l_all[:, n].numpy())
        ref = oracle.attention_unit(q, k, v, row, i, 64, 64, 0.3, False)
        res.append(max(np.abs(got[0] - ref[0]).max(), np.abs(got[1] - ref[1]).max()))
    np.save(os.path.join(out_dir, f"cp{rank}.npy"), np.array([lo, hi, r0, r1] + res))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_exchange_on_gloo_ranks(tmp_path, world):
    mp.start_processes(_cp_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [np.load(tmp_path / f"cp{r}.npy") for r in range(world)]
    import oracle
    from fmha_block_map_gb300 import cp

    # the library's ranges follow the oracle's chunk rule; they tile the kv blocks
    assert cp.kv_shard_bounds(16, world) == oracle.split_bounds(16, world)
    assert [tuple(g[:2].astype(int)) for g in got] == oracle.split_bounds(16, world)
    assert got[-1][3] == 1000 and all(got[r][3] == got[r + 1][2] for r in range(world - 1))
    for g in got:            # every rank combined the gathered partials to the full row
        assert (g[4:] < 1e-10).all()
    with pytest.raises(ValueError):
        cp.kv_shard_bounds(2, 3)


def _rs_worker(rank, world, port, out_dir):
    """Causal context parallelism with the reduce-scatter exchange, on CPU:
    the oracle stands in for this rank's GPU partial (keys of its kv range,
    causal key offset -lo * 64) over every row; scatter_partials_to_owners
    hands each rank the partials of the rows it owns, which it combines."""
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from fmha_block_map_gb300 import cp

    rng = np.random.default_rng(11)
    s, nb = 1000, 16
    q, k = rng.standard_normal((s, 32)), rng.standard_normal((s, 32))
    v = rng.standard_normal((s, 16))
    # a causal LUT: for q block i, a seeded subset of blocks <= i with the diagonal
    luts = [sorted(set(rng.choice(i + 1, size=max(1, (i + 1) // 3), replace=False).tolist())
                   | {i}) for i in range(nb)]
    lo, hi = cp.kv_shard_bounds(nb, world)[rank]
    r0, r1 = cp.shard_rows(s, lo, hi)
    o = np.zeros((s, 16))
    l = np.zeros(s)
    for i in range(nb):
        rows = slice(i * 64, min((i + 1) * 64, s))
        o[rows], l[rows] = oracle.attention_unit(q, k[r0:r1], v[r0:r1],
                                                 oracle.shard_lut_row(luts[i], lo, hi), i, 64,
                                                 64, 0.3, True, key_offset=-lo * 64)
    o_all, l_all, (a, b) = cp.scatter_partials_to_owners(torch.from_numpy(o),
                                                         torch.from_numpy(l))
    got_o, got_l = oracle.combine(o_all.numpy(), l_all.numpy())
    ref_o = np.zeros((s, 16))
    ref_l = np.zeros(s)
    for i in range(nb):
        rows = slice(i * 64, min((i + 1) * 64, s))
        ref_o[rows], ref_l[rows] = oracle.attention_unit(q, k, v, luts[i], i, 64, 64, 0.3, True)
    err = max(np.abs(got_o - ref_o[a:b]).max(), np.abs(got_l - ref_l[a:b]).max())
    np.save(os.path.join(out_dir, f"rs{rank}.npy"), np.array([a, b, o_all.shape[0], err]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_causal_context_parallel_reduce_scatter_on_gloo_ranks(tmp_path, world):
    mp.start_processes(_rs_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [np.load(tmp_path / f"rs{r}.npy") for r in range(world)]
    from fmha_block_map_gb300 import cp

    # the owners' rows tile [0, s) in rank order; each rank combined only its own
    assert [(int(g[0]), int(g[1])) for g in got] == cp.row_owner_bounds(1000, world)
    for g in got:
        assert int(g[2]) == world and g[3] < 1e-10
