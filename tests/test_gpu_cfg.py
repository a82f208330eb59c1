"""CFG merge per codebook + verification on the GPU against the oracle.
Greedy decisions compare the same fp32 merged values on both sides (exact);
sampling decisions are exact outside the 1e-6 margin; TV within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.sampling_parity import assert_pooled_rate, by_request, compare

pytestmark = pytest.mark.gpu


def _run(sv, w, greedy=False):
    got = sv.cfg_merge_sample(w["cond"], w["uncond"], w["cb_id_base"], w["cb_data_offset"], w["S"], w["W"], w["w"],
                              None if greedy else w["draft_logits"], w["R"], w["k"], w["draft"], w["seeds"],
                              w["temperature"])
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in got.items()}


def _oracle(w, greedy=False):
    return oracle.cfg_merge_sample(
        workloads.host_rows(w["cond"]), workloads.host_rows(w["uncond"]), w["cb_id_base"], w["cb_data_offset"],
        w["S"], w["W"], w["w"], None if greedy else workloads.host_rows(w["draft_logits"]), w["R"], w["k"],
        w["draft"].cpu().numpy(), w["seeds"].cpu().numpy().view(np.uint64), w["temperature"].cpu().numpy())


@pytest.mark.parametrize("R,k,S,W,dtype,T", [
    (8, 4, 9, 4096, torch.bfloat16, 1.0),
    (5, 2, 3, 1000, torch.float32, 0.8),     # odd codebook width
    (4, 6, 1, 257, torch.bfloat16, 1.5),
    (3, 3, 16, 2048, torch.bfloat16, 0.6),   # the largest S
    (3, 2, 2, 9000, torch.bfloat16, 1.0),    # wider than 4096: more threads per row
    (2, 2, 2, 16384, torch.float32, 0.9),    # the widest codebook
])
def test_cfg_sampling(sv, R, k, S, W, dtype, T):
    w = workloads.cfg_batch(R, k, S, W, 3.0, T, dtype, seed=R * 31 + S)
    compare(_run(sv, w), _oracle(w))


@pytest.mark.parametrize("dtype,W", [(torch.bfloat16, 4096), (torch.float32, 1000)])
def test_cfg_extreme_temperatures(sv, dtype, W):
    """T = +inf (every codebook id the same weight), 1e30, 1e-4 and 1e-6 (one-hot) beside an
    ordinary and a greedy request, per codebook as the oracle."""
    T = [float("inf"), 1e30, 1e-4, 1e-6, 0.8, 0.0] * 2
    w = workloads.cfg_batch(len(T), 3, 4, W, 3.0, T, dtype, seed=W + 5)
    compare(_run(sv, w), _oracle(w))


def test_cfg_greedy_and_partition_offsets(sv):
    R, k, S, W = 6, 3, 4, 512
    offs = [100 + W * s for s in range(S)]
    w = workloads.cfg_batch(R, k, S, W, 2.5, 0.0, torch.bfloat16, seed=5, row_len=100 + S * W + 37, offsets=offs,
                            greedy_drafts=1.0)
    got, want = _run(sv, w, greedy=True), _oracle(w, greedy=True)
    for key in ("accept_len", "tokens", "status"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    assert np.all(np.isnan(got["tv"]))
    # T > 0 with draft rows, but a NaN in one merged row: that request verifies greedily
    w2 = workloads.cfg_batch(R, k, S, W, 2.5, 1.0, torch.bfloat16, seed=6, row_len=100 + S * W + 37, offsets=offs)
    c = w2["cond"].clone()
    c[(2 * (k + 1) + 1) * S + 2, offs[2] + 9] = float("nan")
    w2["cond"] = c
    compare(_run(sv, w2), _oracle(w2))


def _oracle_par(w):
    """The oracle over every request of a batch, on the host threads."""
    k, S = w["k"], w["S"]
    c, u, y = (workloads.host_rows(w[key]) for key in ("cond", "uncond", "draft_logits"))
    draft = w["draft"].cpu().numpy()
    seeds = w["seeds"].cpu().numpy().view(np.uint64)
    T = w["temperature"].cpu().numpy()
    rr = (k + 1) * S
    return by_request(lambda lo, hi: oracle.cfg_merge_sample(
        c[lo * rr:hi * rr], u[lo * rr:hi * rr], w["cb_id_base"], w["cb_data_offset"], S, w["W"], w["w"],
        y[lo * k * S:hi * k * S], hi - lo, k, draft[lo:hi], seeds[lo:hi], T[lo:hi]), w["R"])


def test_cfg_workload_full_size(sv):
    """The full-size CFG configuration (256 requests x 5 frames x 9 codebooks of 4096) against the
    oracle, then further seeded batches of it until more than 10^5 codebook rows are compared:
    fewer than 1e-5 of the pooled rows may be exempt.  Flat codebooks: most frames are
    rejected early."""
    rows = exempt = b = 0
    while rows < 100_000:
        w = workloads.cfg_workload(batch=b)
        got, want = _run(sv, w), _oracle_par(w)
        exempt += compare(got, want, stats=b % 4 == 0, pooled=True, label=f"cfg batch {b}")
        if b == 0:
            assert want["accept_len"].mean() < 2.0
            ref = _oracle(w)  # the threaded oracle gives the single-threaded oracle's bits
            for key in ("accept_len", "tokens", "status", "tv"):
                np.testing.assert_array_equal(np.nan_to_num(want[key]), np.nan_to_num(ref[key]), err_msg=key)
        rows += w["R"] * (w["k"] + 1) * w["S"]
        b += 1
    assert_pooled_rate(exempt, rows)


def test_near_tie_codebook_races_outside_the_margin(sv):
    """CFG codebook races whose two smallest keys are within 2e-6 .. 1e-4 (relative): outside the
    exempt margin, so the kernel must pick exactly the oracle's token."""
    R, k, S, W = 40_000, 1, 4, 64
    w = workloads.cfg_batch(R, k, S, W, 2.0, 1.0, torch.float32, sigma_h=0.6, bump=1.0, seed=88)
    got, want = _run(sv, w), _oracle_par(w)
    compare(got, want, stats=False)
    rm = want["race_margin"]
    near = ((rm > 2e-6) & (rm < 1e-4)).any(axis=1)
    assert near.sum() >= 5, near.sum()
    for key in ("accept_len", "tokens"):
        np.testing.assert_array_equal(got[key][near], want[key][near], err_msg=key)
