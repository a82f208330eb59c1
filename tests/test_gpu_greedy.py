"""Greedy verification on the GPU against the fp64 CPU oracle, element by
element: accept lengths, tokens, branch and status must be identical (the
decisions compare bf16/fp32 inputs, which is exact in any precision)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.sampling_parity import commits_at_least_one_token

pytestmark = pytest.mark.gpu


def _check(sv, target, R, k, branches, draft, out=None):
    got = sv.verify_greedy(target, R, k, branches, draft, out=out)
    torch.cuda.synchronize()
    want = oracle.verify_greedy(workloads.host_rows(target), R, k, branches, draft.cpu().numpy())
    for key in ("accept_len", "tokens", "branch", "status"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)
    commits_at_least_one_token(want["accept_len"], want["tokens"])
    return got, want


def test_tiny_fp32(sv):
    w = workloads.tiny_greedy()
    _, want = _check(sv, w["target"], w["R"], w["k"], 1, w["draft"])
    assert np.all(want["accept_len"] >= 0)


@pytest.mark.parametrize(
    "R,k,branches,V,dtype,row_pad",
    [
        (5, 8, 1, 4096, torch.bfloat16, 0),
        (7, 3, 2, 4099, torch.bfloat16, 0),     # rows not 16-byte aligned: plain-load path
        (6, 5, 1, 4100, torch.bfloat16, 4),     # aligned rows with a sub-16-byte tail
        (3, 40, 1, 1000, torch.float32, 0),     # k > 32: several ballots
        (2, 7, 2, 151936, torch.bfloat16, 0),
        (3, 4, 1, 151936, torch.float32, 0),
        (1, 0, 1, 5000, torch.bfloat16, 0),     # k = 0: one autoregressive step
        (9, 2, 1, 17, torch.float32, 3),        # tiny vocabulary
        (4, 33, 2, 3001, torch.bfloat16, 7),
        (2, 256, 1, 300, torch.bfloat16, 0),    # largest k
        (40, 6, 2, 65536, torch.bfloat16, 0),
    ],
)
def test_random_shapes(sv, R, k, branches, V, dtype, row_pad):
    w = workloads.greedy_batch(R, k, V, dtype, branches=branches, p_full=0.5, p_first=0.5, seed=R * 1000 + k,
                               row_pad=row_pad)
    _check(sv, w["target"], R, k, branches, w["draft"])


@pytest.mark.parametrize("R,k,branches,V,dtype", [
    (9, 5, 4, 4096, torch.bfloat16),
    (6, 3, 8, 151936, torch.bfloat16),
    (5, 7, 3, 3001, torch.float32),     # plain-load path
])
def test_tree_drafts(sv, R, k, branches, V, dtype):
    """More than two branches sharing the first row (tree drafts), also with the top-2 output."""
    w = workloads.greedy_batch(R, k, V, dtype, branches=branches, p_full=0.5, p_first=0.5, seed=R * 31 + branches)
    got, want = _check(sv, w["target"], R, k, branches, w["draft"])
    assert len(set(want["branch"].tolist())) > 1  # the winning branch varies
    _check_top2(sv, w["target"], R, k, branches, w["draft"])


def test_ties_go_to_lowest_index(sv):
    g = torch.Generator(device="cuda").manual_seed(5)
    R, k, V = 6, 5, 3000
    z = torch.randint(0, 3, (R * (k + 1), V), generator=g, device="cuda").to(torch.bfloat16)
    host = workloads.host_rows(z)
    widened = (host.astype(np.uint32) << 16).view(np.float32)
    first = np.argmax(widened, axis=1).reshape(R, k + 1)  # numpy: first index of the maximum
    draft = first[:, :k].copy()
    draft[1, 2] = (draft[1, 2] + 1) % V
    draft[3, 0] = V - 1
    d = torch.from_numpy(draft.astype(np.int32)).view(R, 1, k).cuda()
    _check(sv, z, R, k, 1, d)


def test_nan_inf_and_out_of_range(sv):
    R, k, V = 5, 4, 2048
    w = workloads.greedy_batch(R, k, V, torch.float32, branches=1, p_full=1.0, seed=77)
    t = w["target"].clone()
    t[0, 10] = float("nan")                 # NaN in request 0
    t[6, :] = float("nan")                  # an all-NaN row in request 1
    t[11, 100] = float("inf")               # +inf in request 2 becomes its argmax
    t[16, :] = float("-inf")                # all -inf row in request 3
    t[21, ::2] = float("nan")
    d = w["draft"].clone()
    d[4, 0, 1] = -3
    d[4, 0, 2] = V + 11
    _check(sv, t, R, k, 1, d)


def test_listen_full_size_and_determinism(sv):
    w = workloads.listen()
    got, want = _check(sv, w["target"], w["R"], w["k"], 2, w["draft"])
    # 95% of main branches match fully; position-0 mismatches fall back to the runner-up
    assert (want["accept_len"] == 32).mean() > 0.8
    again = sv.verify_greedy(w["target"], w["R"], w["k"], 2, w["draft"])
    torch.cuda.synchronize()
    for key in ("accept_len", "tokens", "branch", "status"):
        assert torch.equal(got[key], again[key])


def test_strided_bf16_rows_and_reused_workspace(sv):
    R, k, V = 16, 6, 151936
    w = workloads.greedy_batch(R, k, V, torch.bfloat16, branches=2, p_full=0.6, seed=3, row_pad=64)
    ws = torch.empty(sv.verify_greedy_workspace(R, k, 2, V), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        got = sv.verify_greedy(w["target"], R, k, 2, w["draft"], workspace=ws)
    torch.cuda.synchronize()
    want = oracle.verify_greedy(workloads.host_rows(w["target"]), R, k, 2, w["draft"].cpu().numpy())
    np.testing.assert_array_equal(got["tokens"].cpu().numpy(), want["tokens"])


def test_zero_requests_is_a_no_op(sv):
    t = torch.zeros(0, 100, device="cuda", dtype=torch.bfloat16)
    out = dict(accept_len=torch.full((1,), 7, dtype=torch.int32, device="cuda"),
               tokens=torch.full((1, 3), 7, dtype=torch.int32, device="cuda"))
    sv.verify_greedy(t, 0, 2, 1, torch.zeros(0, 1, 2, dtype=torch.int32, device="cuda"), out=out)
    torch.cuda.synchronize()
    assert out["accept_len"].item() == 7


def test_accept_scan_matches_oracle(sv):
    g = np.random.default_rng(3)
    for R, k in [(1, 1), (37, 7), (5, 70), (3, 256)]:
        acc = (g.random((R, k)) < 0.85).astype(np.uint8)
        draft = g.integers(0, 5000, (R, k)).astype(np.int32)
        fix = g.integers(0, 5000, (R, k + 1)).astype(np.int32)
        got = sv.accept_scan(torch.from_numpy(acc).cuda(), torch.from_numpy(draft).cuda(),
                             torch.from_numpy(fix).cuda())
        torch.cuda.synchronize()
        want = oracle.accept_scan(acc, draft, fix)
        np.testing.assert_array_equal(got["accept_len"].cpu().numpy(), want["accept_len"])
        np.testing.assert_array_equal(got["tokens"].cpu().numpy(), want["tokens"])


# --------------------------------------------------------------------------
# argmax and runner-up of every row, fused into the greedy pass
# --------------------------------------------------------------------------
def _check_top2(sv, target, R, k, branches, draft):
    got = sv.verify_greedy_top2(target, R, k, branches, draft)
    torch.cuda.synchronize()
    host = workloads.host_rows(target)
    want = oracle.verify_greedy(host, R, k, branches, draft.cpu().numpy())
    for key in ("accept_len", "tokens", "branch", "status"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)
    np.testing.assert_array_equal(got["top2"].cpu().numpy(), oracle.top2_rows(host), err_msg="top2")
    return got


@pytest.mark.parametrize(
    "R,k,branches,V,dtype,row_pad",
    [
        (5, 8, 1, 4096, torch.bfloat16, 0),
        (7, 3, 2, 4099, torch.bfloat16, 0),     # plain-load path
        (6, 5, 1, 4100, torch.bfloat16, 4),     # sub-16-byte tail
        (3, 4, 1, 151936, torch.float32, 0),
        (2, 7, 2, 151936, torch.bfloat16, 0),   # several segments per row
        (9, 2, 1, 17, torch.float32, 3),        # tiny vocabulary
        (4, 1, 1, 7, torch.bfloat16, 1),        # fewer ids than a vector
        (40, 6, 2, 65536, torch.bfloat16, 0),
    ],
)
def test_top2_random_shapes(sv, R, k, branches, V, dtype, row_pad):
    w = workloads.greedy_batch(R, k, V, dtype, branches=branches, p_full=0.5, p_first=0.5, seed=R * 77 + k,
                               row_pad=row_pad)
    _check_top2(sv, w["target"], R, k, branches, w["draft"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_top2_ties_nan_and_inf(sv, dtype):
    """Values from a small set (ties everywhere), NaN, +inf, all -inf and all-NaN rows."""
    g = torch.Generator(device="cuda").manual_seed(9)
    R, k, V = 6, 5, 3001
    z = torch.randint(-2, 3, (R * (k + 1), V), generator=g, device="cuda").to(dtype)
    z[0, 5] = float("nan")
    z[1, ::3] = float("nan")
    z[2, 77] = float("inf")
    z[3, 100] = float("inf")
    z[3, 2000] = float("inf")                # tied +inf
    z[4, :] = float("-inf")
    z[5, :] = float("nan")
    z[6, :] = float("-inf")
    z[6, 2999] = 1.0                         # one finite value, the rest -inf
    z[7, :] = 2.0                            # a constant row
    z[8, 1] = 50.0                           # a unique maximum, the runner-up tied many times
    d = torch.zeros(R, 1, k, dtype=torch.int32, device="cuda")
    _check_top2(sv, z, R, k, 1, d)


def test_top2_one_id_rows(sv):
    z = torch.tensor([[3.0], [float("nan")], [-1.0]], device="cuda", dtype=torch.float32)
    got = _check_top2(sv, z, 3, 0, 1, torch.zeros(3, 1, 0, dtype=torch.int32, device="cuda"))
    assert got["top2"][:, 1].tolist() == [-1, -1, -1]


def test_top2_listen_runner_up(sv):
    """On the listen workload a runner-up branch whose main branch starts with the argmax of
    row 0 starts from the second-best id of row 0."""
    w = workloads.listen()
    got = _check_top2(sv, w["target"], w["R"], w["k"], 2, w["draft"])
    rows_per = 2 * w["k"] + 1
    first0 = got["top2"].view(w["R"], rows_per, 2)[:, 0, 0]
    second0 = got["top2"].view(w["R"], rows_per, 2)[:, 0, 1]
    main = w["draft"][:, 0, 0] == first0
    assert main.sum() > w["R"] // 2
    assert torch.equal(second0[main], w["draft"][main, 1, 0])


# --------------------------------------------------------------------------
# modality of a row: the vocabulary partition of its unmasked argmax
# --------------------------------------------------------------------------
def _va_partitions(V=151936, S=9, W=4096):
    text = V - S * W
    return [0, text] + [text + W * (s + 1) for s in range(S)]


@pytest.mark.parametrize("dtype,N,V,starts", [
    (torch.bfloat16, 300, 151936, _va_partitions()),       # the text part, then 9 codebooks of 4096
    (torch.float32, 70, 151936, _va_partitions()),
    (torch.bfloat16, 40, 5003, [0, 1000, 1000, 2500, 4096]),  # an empty partition, ids past the last
    (torch.float32, 9, 17, [3, 9]),                        # ids before the first partition
    (torch.bfloat16, 50, 65536, list(range(0, 65537, 1024))),  # the most partitions (64)
])
def test_infer_modality_matches_oracle(sv, dtype, N, V, starts):
    g = torch.Generator(device="cuda").manual_seed(N + V)
    z = torch.randn(N, V, generator=g, device="cuda") * 3.0
    # plant the maximum in a random partition (or none) for most rows
    pick = torch.randint(0, V, (N,), generator=g, device="cuda")
    z[torch.arange(N, device="cuda"), pick] = 40.0
    z = z.to(dtype)
    z[0, :] = float("nan")                                 # argmax 0, flagged
    if V > 2000:
        b = starts[1]
        z[1, b - 1] = z[1, b] = 60.0                       # a tie across a partition boundary
        z[2, 7] = float("inf")                             # +inf maximum, flagged
    got = sv.infer_modality(z, starts)
    torch.cuda.synchronize()
    want = oracle.infer_modality(workloads.host_rows(z), np.array(starts, np.int32))
    for key in ("amax", "part", "mask_lo", "mask_hi"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)
    st = got["status"].cpu().numpy()
    assert st[0] & oracle.ST_BAD_LOGITS
    if V > 2000:
        assert st[2] & oracle.ST_BAD_LOGITS and not (st[3:] & oracle.ST_BAD_LOGITS).any()
