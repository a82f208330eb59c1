"""The N > 1 path on CPU: two gloo ranks.  Requests are independent and every
result is a function of (seed, row, id), so sharding a batch by request across
ranks and gathering the outputs gives the single-rank result; the benchmark's
rank plumbing (process group, barrier, max over ranks) runs on gloo."""
import json
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import oracle
    import workloads

    w_, r_, _ = bench._dist()  # gloo: no GPU here
    assert (w_, r_) == (world, rank) and dist.get_backend() == "gloo"
    # timing plumbing: every rank contributes its own time, all see the maximum
    assert bench._max_over_ranks(1.5 + rank, world, "cpu") == 1.5 + world - 1
    bench._barrier(world)

    w = workloads.tiny_sample(device="cpu")
    R, k = w["R"], w["k"]
    lo, hi = rank * R // world, (rank + 1) * R // world
    target = workloads.host_rows(w["target"])[lo * (k + 1):hi * (k + 1)]
    draft_logits = workloads.host_rows(w["draft_logits"])[lo * k:hi * k]
    out = oracle.verify_sample(target, draft_logits, None, hi - lo, k, w["draft"].numpy()[lo:hi],
                               w["seeds"].numpy()[lo:hi], w["temperature"].numpy()[lo:hi])
    g = workloads.tiny_greedy(device="cpu")
    gt = workloads.host_rows(g["target"])[lo * (k + 1):hi * (k + 1)]
    gout = oracle.verify_greedy(gt, hi - lo, k, 1, g["draft"].numpy()[lo:hi])
    shard = {key: out[key].tolist() for key in ("accept_len", "tokens", "tv", "status")}
    shard.update({"g_" + key: gout[key].tolist() for key in ("accept_len", "tokens")})
    parts = [None] * world
    dist.all_gather_object(parts, shard)
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(parts, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_request(tmp_path):
    torch_mp = pytest.importorskip("torch.multiprocessing")
    import oracle
    import workloads

    out_path = str(tmp_path / "parts.json")
    torch_mp.spawn(_rank_main, args=(2, _free_port(), out_path), nprocs=2, join=True)
    parts = json.load(open(out_path))

    w = workloads.tiny_sample(device="cpu")
    R, k = w["R"], w["k"]
    full = oracle.verify_sample(workloads.host_rows(w["target"]), workloads.host_rows(w["draft_logits"]), None, R,
                                k, w["draft"].numpy(), w["seeds"].numpy(), w["temperature"].numpy())
    g = workloads.tiny_greedy(device="cpu")
    gfull = oracle.verify_greedy(workloads.host_rows(g["target"]), R, k, 1, g["draft"].numpy())
    for key in ("accept_len", "tokens", "status"):
        np.testing.assert_array_equal(np.concatenate([np.asarray(p[key]) for p in parts]), full[key], err_msg=key)
    np.testing.assert_array_equal(np.concatenate([np.asarray(p["tv"]) for p in parts]), full["tv"])
    for key in ("accept_len", "tokens"):
        np.testing.assert_array_equal(np.concatenate([np.asarray(p["g_" + key]) for p in parts]), gfull[key])
