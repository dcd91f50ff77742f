"""Rank bodies of the two-process CPU (gloo) tests in test_multirank.py.  Each
function runs in a spawned process; failures surface as a non-zero exit."""

import os

import numpy as np
import torch
import torch.distributed as dist


def _init(rank: int, world: int, port: int):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    os.environ["LOCAL_RANK"] = str(rank)


def bench_helpers(rank: int, world: int, port: int, port2: int, out_dir: str):
    """bench.py's multi-rank plumbing: rendezvous from the environment, the
    max of the ranks' times, the barrier, and the reference arm leaving
    without work on ranks other than 0."""
    _init(rank, world, port)
    import bench
    w, r, local, pg = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank) and pg is not None
    v = bench.max_over_ranks(1.5 + rank, pg)
    bench.barrier(pg)
    with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as f:
        f.write(repr(v))
    dist.destroy_process_group()
    # the reference arm: every rank joins the rendezvous, only rank 0 works
    _init(rank, world, port2)
    if rank == 0:
        bench.dist_setup(None)
    else:
        class Args:  # nothing is read before a rank other than 0 returns
            pass
        assert bench.run_reference(Args()) is None
        with open(os.path.join(out_dir, f"ref{rank}.txt"), "w") as f:
            f.write("returned")
    dist.barrier()
    dist.destroy_process_group()


def ep_tp_switch(rank: int, world: int, port: int, out_dir: str):
    """A whole EP -> TP -> EP expert-weight switch over `world` ranks: the
    local pack, one all-to-all, and a check that every rank then holds the TP
    layout (E, 2I/P, H) / (E, H, I/P) of all experts; then the way back (the
    all-to-all, then the local unpack) restores each rank's experts."""
    _init(rank, world, port)
    import oracle
    dist.init_process_group("gloo")
    P = world
    E, H, I = 4, 8, 16
    E_l, Ip = E // P, I // P
    rng = np.random.default_rng(0)  # the same global weights on every rank
    W13 = rng.integers(-2**31, 2**31 - 1, size=(E, 2 * I, H), dtype=np.int64).astype(np.int32)
    W2 = rng.integers(-2**31, 2**31 - 1, size=(E, H, I), dtype=np.int64).astype(np.int32)
    mine = slice(rank * E_l, (rank + 1) * E_l)  # EP: this rank's complete experts
    c13, c2 = oracle.reshard_pack(W13[mine], W2[mine], P)
    r13, r2 = torch.empty(c13.shape, dtype=torch.int32), torch.empty(c2.shape, dtype=torch.int32)
    dist.all_to_all_single(r13, torch.from_numpy(c13))
    dist.all_to_all_single(r2, torch.from_numpy(c2))
    # received chunk q = peer q's experts, this rank's slice: the TP layout
    tp13 = r13.numpy().reshape(E, 2 * Ip, H)
    tp2 = r2.numpy().reshape(E, H, Ip)
    gate = W13[:, rank * Ip:(rank + 1) * Ip]
    up = W13[:, I + rank * Ip:I + (rank + 1) * Ip]
    assert np.array_equal(tp13, np.concatenate([gate, up], axis=1))
    assert np.array_equal(tp2, W2[:, :, rank * Ip:(rank + 1) * Ip])
    # TP -> EP: this rank's shard of peer q's experts is contiguous in the TP
    # layout, so the all-to-all goes first, then the local unpack
    b13, b2 = torch.empty_like(r13), torch.empty_like(r2)
    dist.all_to_all_single(b13, torch.from_numpy(np.ascontiguousarray(tp13)))
    dist.all_to_all_single(b2, torch.from_numpy(np.ascontiguousarray(tp2)))
    e13, e2 = oracle.reshard_unpack(b13.numpy(), b2.numpy(), P)
    assert np.array_equal(e13, W13[mine]) and np.array_equal(e2, W2[mine])
    with open(os.path.join(out_dir, f"ok{rank}.txt"), "w") as f:
        f.write("ok")
    dist.destroy_process_group()
