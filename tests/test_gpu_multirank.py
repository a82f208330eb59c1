"""The N > 1 path with the library itself: two gloo ranks, both on the visible GPU, each verify
their half of one batch through the CUDA library (sampling with a d2t draft vocabulary, and
greedy speculative-listening verification); the gathered halves equal the single-process call
bit for bit, because every output is a function of the request's own inputs.  The ranks' kernels
never wait on one another: each rank's calls are independent, and only the host gathers."""
import json
import os
import socket

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _sample_batch():
    T = [0.7 if r % 3 else 0.0 for r in range(24)]
    return workloads.sample_batch(24, 7, workloads.V_QWEN, workloads.VD_DRAFT, torch.bfloat16, T=T, sigma_pos=0.8,
                                  delta=2.7, seed=53, seed_base=211)


def _greedy_batch():
    return workloads.listen(R=6, seed=97)


def _bits(t):
    a = t.cpu().numpy()
    return (a.view(np.uint32) if a.dtype == np.float32 else a).tolist()


def _sample_call(sv, w, lo, hi):
    k = w["k"]
    got = sv.verify_sample(w["target"][lo * (k + 1):hi * (k + 1)], w["draft_logits"][lo * k:hi * k], w["d2t"],
                           hi - lo, k, w["draft"][lo:hi], w["seeds"][lo:hi], w["temperature"][lo:hi])
    torch.cuda.synchronize()
    return {key: _bits(v) for key, v in got.items()}


def _greedy_call(sv, w, lo, hi):
    rpr = 1 + w["branches"] * w["k"]
    got = sv.verify_greedy(w["target"][lo * rpr:hi * rpr], hi - lo, w["k"], w["branches"], w["draft"][lo:hi])
    torch.cuda.synchronize()
    return {key: _bits(v) for key, v in got.items()}


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import serving_sampler_gb300 as sv

    dist.init_process_group("gloo", rank=rank, world_size=world)
    sv.load()  # built in-tree by the parent process
    w, g = _sample_batch(), _greedy_batch()
    lo, hi = rank * w["R"] // world, (rank + 1) * w["R"] // world
    glo, ghi = rank * g["R"] // world, (rank + 1) * g["R"] // world
    shard = {"sample": _sample_call(sv, w, lo, hi), "greedy": _greedy_call(sv, g, glo, ghi)}
    parts = [None] * world
    dist.all_gather_object(parts, shard)
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(parts, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_library_calls(sv, tmp_path):
    torch_mp = pytest.importorskip("torch.multiprocessing")
    out_path = str(tmp_path / "parts.json")
    torch_mp.spawn(_rank_main, args=(2, _free_port(), out_path), nprocs=2, join=True)
    parts = json.load(open(out_path))
    w, g = _sample_batch(), _greedy_batch()
    full = {"sample": _sample_call(sv, w, 0, w["R"]), "greedy": _greedy_call(sv, g, 0, g["R"])}
    for call in ("sample", "greedy"):
        for key, v in full[call].items():
            gathered = np.concatenate([np.asarray(p[call][key]) for p in parts])
            np.testing.assert_array_equal(gathered, np.asarray(v), err_msg=f"{call} {key}")
    # the gathered sampling batch holds sampled and greedily verified requests
    T = w["temperature"].cpu().numpy()
    assert (T > 0).any() and (T <= 0).any()
