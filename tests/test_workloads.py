"""The synthetic inputs have the statistics the workload descriptions give (CPU).

The listen drafts follow the speculative-listening observations (95% of main
drafts match fully, 88% of the mismatches at the first position), the planted
ids are the rows' argmaxes, the d2t drafter's acceptance falls from about 0.7 to
about 0.4 along the draft, and the CFG rows are flat (guided top-1 near 0.2).
Results come from the oracle or from plain numpy on the generated inputs."""
import numpy as np
import torch

import oracle
import workloads


def test_listen_drafts_follow_the_observed_match_profile():
    R, k = 4000, 32
    w = workloads.greedy_batch(R, k, 512, torch.bfloat16, 3.0, branches=2, seed=1236, device="cpu")
    main = w["draft"][:, 0].numpy()
    top = w["planted"].numpy()
    miss = main != top[:, :k]
    full = ~miss.any(axis=1)
    first_pos = miss.argmax(axis=1)
    se = lambda p, n: 4 * np.sqrt(p * (1 - p) / n)
    assert abs(full.mean() - 0.95) < se(0.95, R)
    at0 = (first_pos[~full] == 0).mean()
    assert abs(at0 - 0.88) < se(0.88, (~full).sum())
    # the runner-up branch starts with the best token other than the main draft's first
    runner = w["draft"][:, 1].numpy()
    assert np.all(runner[:, 0] != main[:, 0])
    assert np.all(runner[main[:, 0] != top[:, 0], 0] == top[main[:, 0] != top[:, 0], 0])


def test_planted_ids_are_the_argmax_of_bf16_rows():
    w = workloads.greedy_batch(6, 4, 151936, torch.bfloat16, 3.0, branches=2, seed=3, device="cpu")
    rows = workloads.host_rows(w["target"])
    top2 = oracle.top2_rows(rows)
    assert np.array_equal(top2[:, 0], w["planted"].numpy().reshape(-1))
    # the runner-up of each request's shared first row is the planted second best
    main = w["draft"][:, 0].numpy()
    second = top2.reshape(6, -1, 2)[:, 0, 1]
    ok = main[:, 0] == w["planted"].numpy()[:, 0]
    assert np.array_equal(w["draft"][:, 1].numpy()[ok, 0], second[ok])


def test_d2t_drafter_acceptance_falls_along_the_draft():
    R = 6
    w = workloads.sample_batch(R, 7, workloads.V_QWEN, workloads.VD_DRAFT, torch.bfloat16, T=0.7,
                               sigma_pos=workloads.D2T_SIGMA, delta=workloads.D2T_DELTA, z_sigma=3.0, seed=1237,
                               seed_base=1234, device="cpu")
    out = oracle.verify_sample(workloads.host_rows(w["target"]), workloads.host_rows(w["draft_logits"]),
                               w["d2t"].numpy(), R, 7, w["draft"].numpy(), w["seeds"].numpy().view(np.uint64),
                               w["temperature"].numpy())
    alpha = 1 - out["tv"].mean(axis=0)
    assert 0.6 < alpha[0] < 0.8 and 0.3 < alpha[-1] < 0.5
    assert alpha[0] > alpha[3] > alpha[-1]


def test_cfg_rows_are_flat():
    w = workloads.cfg_batch(4, 4, 9, 4096, 3.0, 1.0, torch.float32, seed=1238, device="cpu")
    c = w["cond"].numpy().astype(np.float64)
    u = w["uncond"].numpy().astype(np.float64)
    m = u + 3.0 * (c - u)
    p = np.exp(m - m.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert 0.12 < p.max(axis=1).mean() < 0.3
