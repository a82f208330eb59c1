"""The hypothesis pool on the GPU against the CPU oracle: pool contents, used
lengths, status, match lengths and continuations must be identical."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _append_both(sv, pool_d, plen_d, pool_h, plen_h, drafts):
    st = torch.full((pool_d.shape[0],), -5, dtype=torch.int32, device="cuda")
    sv.pool_append(pool_d, plen_d, _dev(drafts), status=st)
    want = oracle.pool_append(pool_h, plen_h, drafts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(plen_d.cpu().numpy(), want["pool_len"], err_msg="pool_len")
    np.testing.assert_array_equal(st.cpu().numpy(), want["status"], err_msg="status")
    used = want["pool_len"]
    got_pool = pool_d.cpu().numpy()
    for r in range(len(used)):
        np.testing.assert_array_equal(got_pool[r, :used[r]], want["pool"][r, :used[r]], err_msg=f"pool row {r}")
    return want["pool"], want["pool_len"]


def _lookup_both(sv, pool_h, plen_h, suffix, gamma, pool_d=None, plen_d=None):
    pool_d = _dev(pool_h) if pool_d is None else pool_d
    plen_d = _dev(plen_h) if plen_d is None else plen_d
    got = sv.pool_lookup(pool_d, plen_d, _dev(suffix), gamma)
    want = oracle.pool_lookup(pool_h, plen_h, suffix, gamma)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["match_len"].cpu().numpy(), want["match_len"], err_msg="match_len")
    np.testing.assert_array_equal(got["cont"].cpu().numpy(), want["cont"], err_msg="cont")
    return want


def test_session_workload(sv):
    w = workloads.pool_session()
    R, Lp = w["R"], w["Lp"]
    pool_h = np.full((R, Lp), -3, np.int32)
    plen_h = np.zeros(R, np.int32)
    pool_d = _dev(pool_h)
    plen_d = _dev(plen_h)
    for c, d in enumerate(w["drafts"]):
        pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, d)
        if c % 6 == 5:  # look up between chunks too
            _lookup_both(sv, pool_h, plen_h, w["suffix"], w["gamma"], pool_d, plen_d)
    want = _lookup_both(sv, pool_h, plen_h, w["suffix"], w["gamma"], pool_d, plen_d)
    assert (want["match_len"] > 0).sum() >= 10  # the workload exercises real matches


@pytest.mark.parametrize(
    "R,Lp,vocab,N,gamma,seed",
    [
        (300, 2000, 3, 5, 33, 1),      # more requests than SMs; matches everywhere, many ties
        (7, 20000, 4, 64, 256, 2),     # long pools (many strides of the block), longest suffix, widest gamma
        (16, 600, 50, 1, 1, 3),        # unigram matches only
        (16, 600, 2, 8, 0, 4),         # gamma 0: the match length alone
        (5, 0, 3, 4, 8, 5),            # capacity 0
        (9, 97, 6, 0, 8, 6),           # N 0: never a match
    ],
)
def test_random_pools(sv, R, Lp, vocab, N, gamma, seed):
    rng = np.random.default_rng(seed)
    pool = np.full((R, Lp), -1, np.int32)
    plen = np.zeros(R, np.int32)
    for r in range(R):
        pos = 0
        while Lp > 0:
            n = int(rng.integers(1, 40))
            if pos + n + 1 > Lp:
                break
            pool[r, pos:pos + n] = rng.integers(0, vocab, n)
            pos += n + 1
        plen[r] = pos
        pool[r, pos:] = rng.integers(0, vocab, Lp - pos)  # unused entries hold tokens: never read
    suffix = rng.integers(0, vocab, (R, N)).astype(np.int32)
    for r in range(0, R, 4):  # shorter outputs
        suffix[r, :int(rng.integers(0, N + 1))] = -1
    want = _lookup_both(sv, pool, plen, suffix, gamma)
    if Lp > 0 and N > 0:
        assert want["match_len"].max() > 0


def test_pool_len_outside_the_capacity(sv):
    pool = np.array([[5, 6, 7, -1, 5, 9, -1, 8]] * 6, np.int32)
    plen = np.array([-9, 0, 2, 5, 8, 1 << 20], np.int32)
    suffix = np.array([[5]] * 6, np.int32)
    _lookup_both(sv, pool, plen, suffix, 4)
    # append: a used length outside [0, Lp] reads as a full pool
    drafts = np.array([[1, 2]] * 6, np.int32)
    pool_d, plen_d = _dev(pool), _dev(plen)
    _append_both(sv, pool_d, plen_d, pool, plen, drafts)


def test_pool_full_and_early_ends(sv):
    R, Lp = 4, 12
    pool_h = np.full((R, Lp), -2, np.int32)
    plen_h = np.array([0, 3, 7, 12], np.int32)
    pool_d, plen_d = _dev(pool_h), _dev(plen_h)
    drafts = np.array([[1, 2, 3, 4, -1, 5], [9, -1, 7, 7, 7, 7], [-1, 1, 1, 1, 1, 1], [1, 2, 3, 4, 5, 6]], np.int32)
    pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, drafts)
    assert plen_h.tolist() == [5, 5, 7, 12]
    big = np.arange(R * 6, dtype=np.int32).reshape(R, 6)
    pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, big)
    assert plen_h.tolist() == [12, 12, 7, 12]


def test_case_study_pool(sv):
    # drafts of the tool-call case study: the call drafted in chunk 2, redrafted and cut off in chunk 3
    OK, SURE, CALL, FIND, LP, TYO, COMMA, FRI, RP, END = 20, 21, 10, 11, 12, 13, 14, 15, 16, 17
    drafts = [[OK], [SURE, CALL, FIND, LP, TYO, COMMA, FRI, RP, END], [CALL, FIND, LP, TYO], [OK]]
    pool_h = np.zeros((1, 19), np.int32)
    plen_h = np.zeros(1, np.int32)
    pool_d, plen_d = _dev(pool_h), _dev(plen_h)
    for d in drafts:
        row = np.full((1, 9), -1, np.int32)
        row[0, :len(d)] = d
        pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, row)
    suffix = np.array([[SURE, CALL, FIND, LP]], np.int32)
    want = _lookup_both(sv, pool_h, plen_h, suffix, 8, pool_d, plen_d)
    assert want["cont"][0, :5].tolist() == [TYO, COMMA, FRI, RP, END]


def test_empty_batch(sv):
    pool = torch.zeros((0, 16), dtype=torch.int32, device="cuda")
    plen = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = sv.pool_lookup(pool, plen, torch.zeros((0, 4), dtype=torch.int32, device="cuda"), 8)
    sv.pool_append(pool, plen, torch.zeros((0, 4), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert out["match_len"].numel() == 0


@pytest.mark.parametrize("R,N,k", [(300, 8, 7), (5, 64, 256), (9, 1, 0), (7, 40, 33)])
def test_suffix_append(sv, R, N, k):
    rng = np.random.default_rng(R + N + k)
    suffix = rng.integers(0, 1000, (R, N)).astype(np.int32)
    suffix[::3, : N // 2] = -1  # shorter outputs
    tokens = rng.integers(0, 1000, (R, k + 1)).astype(np.int32)
    acc = rng.integers(-2, k + 3, R).astype(np.int32)  # also outside [0, k]: clamped
    for r in range(R):
        tokens[r, max(0, min(acc[r], k)) + 1:] = -1
    s_d = _dev(suffix)
    sv.suffix_append(s_d, _dev(tokens), _dev(acc))
    want = oracle.suffix_append(suffix, tokens, acc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s_d.cpu().numpy(), want)


def test_verify_suffix_lookup_loop_on_the_device(sv):
    # the device-resident loop of the pages' steps 3-5: greedy verification of drafts taken
    # from the pool, the suffix update from its outputs, the next lookup, all on the GPU
    import workloads as wl

    w = wl.greedy_batch(16, 6, 4096, torch.bfloat16, branches=1, p_full=0.5, p_first=0.2, seed=5)
    R, k = w["R"], w["k"]
    drafts = w["draft"].view(R, k)
    pool_h = np.zeros((R, 64), np.int32)
    plen_h = np.zeros(R, np.int32)
    pool_d, plen_d = _dev(pool_h), _dev(plen_h)
    pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, drafts.cpu().numpy())
    out = sv.verify_greedy(w["target"], R, k, 1, w["draft"])
    suffix_h = np.full((R, 8), -1, np.int32)
    s_d = _dev(suffix_h)
    sv.suffix_append(s_d, out["tokens"], out["accept_len"])
    got = sv.pool_lookup(pool_d, plen_d, s_d, k)
    torch.cuda.synchronize()
    tok, acc = out["tokens"].cpu().numpy(), out["accept_len"].cpu().numpy()
    suffix_w = oracle.suffix_append(suffix_h, tok, acc)
    np.testing.assert_array_equal(s_d.cpu().numpy(), suffix_w)
    want = oracle.pool_lookup(pool_h, plen_h, suffix_w, k)
    np.testing.assert_array_equal(got["match_len"].cpu().numpy(), want["match_len"])
    np.testing.assert_array_equal(got["cont"].cpu().numpy(), want["cont"])
