"""Multi-rank host logic on the CPU: two processes over gloo (127.0.0.1).

- bench.py's N > 1 plumbing (rendezvous from the environment, max of the
  ranks' times, barrier, the reference arm's other ranks leaving at once);
- the EP <-> TP expert-weight switch of Moebius (section 3.1 "Weights
  Resharding", Figure 4) end to end with a real all-to-all: the local pack's
  chunk layout lands every shard in the TP layout, and the way back restores
  the experts.  The local permute is the oracle's (the CUDA permute is checked
  against it bit for bit on the GPU)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import multirank_worker as worker


def _port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_bench_multirank_helpers(tmp_path):
    mp.spawn(worker.bench_helpers, args=(2, _port(), _port(), str(tmp_path)), nprocs=2,
             join=True)
    for r in range(2):
        assert float((tmp_path / f"max{r}.txt").read_text()) == 2.5
    assert (tmp_path / "ref1.txt").read_text() == "returned"


@pytest.mark.parametrize("world", [2, 4])
def test_ep_tp_switch_over_all_to_all(tmp_path, world):
    mp.spawn(worker.ep_tp_switch, args=(world, _port(), str(tmp_path)), nprocs=world, join=True)
    assert all((tmp_path / f"ok{r}.txt").exists() for r in range(world))
