"""CPU tests of the parity helper: which rows are exempt, the row-rate rule, and that a
request differing from the oracle passes only when one of its rows is exempt."""
import numpy as np
import pytest

from tests.sampling_parity import EXEMPT_RATE, MARGIN, compare, exempt_rows


def _want(R, k, S=None):
    shape = (R, k + 1) if S is None else (R, k + 1, S)
    tok = np.full(shape, -1, np.int32)
    n = np.zeros(R, np.int32)
    tok[:, 0] = 7
    am = np.full((R, k) if S is None else (R, k, S), np.inf)
    rm = np.full(R if S is None else (R, S), np.inf)
    return dict(accept_len=n, tokens=tok, accept_margin=am, race_margin=rm, status=np.zeros(R, np.int32))


def test_exempt_rows_sampling():
    w = _want(3, 3)
    w["accept_len"][:] = [1, 2, 3]
    for r, n in enumerate(w["accept_len"]):
        w["tokens"][r, : n + 1] = 5
    w["accept_margin"][0, 1] = MARGIN / 2   # a tested position
    w["race_margin"][1] = MARGIN / 3        # the residual race ran on row 2
    w["race_margin"][2] = MARGIN * 2        # not below the margin
    m = exempt_rows(w)
    assert m.shape == (3, 4)
    assert sorted(zip(*np.nonzero(m))) == [(0, 1), (1, 2)]
    w["race_margin"][2] = MARGIN / 2        # the bonus race ran on row k = 3
    assert exempt_rows(w)[2, 3]
    w["accept_margin"][1, 2] = 0.0          # the same row twice counts once
    assert exempt_rows(w).sum() == 3


def test_exempt_rows_cfg_counts_codebook_rows():
    R, k, S = 2, 2, 3
    w = _want(R, k, S)
    w["accept_len"][:] = [0, 2]
    w["race_margin"][0, 2] = 0.0            # frame 0, codebook 2
    w["race_margin"][1, 0] = 0.0            # bonus frame 2, codebook 0
    w["accept_margin"][1, 1, 1] = 0.0       # frame 1, codebook 1
    m = exempt_rows(w).reshape(R, k + 1, S)
    assert sorted(zip(*np.nonzero(m))) == [(0, 0, 2), (1, 1, 1), (1, 2, 0)]


def test_compare_rules():
    R, k = 40_000, 1  # 80,000 rows: one exempt row is 1.25e-5 of them, above the rate
    want = _want(R, k)
    got = {key: v.copy() for key, v in want.items()}
    compare(got, want, stats=False, label="plain", log=False)
    got["tokens"][3, 0] = 9                 # a request differs without an exempt row
    with pytest.raises(AssertionError, match="differ"):
        compare(got, want, stats=False, label="differs", log=False)
    want["accept_margin"][3, 0] = 0.0       # now its row is exempt, but 1 / 80,000 >= 1e-5
    assert 1 >= EXEMPT_RATE * R * (k + 1)
    with pytest.raises(AssertionError, match="exempt rows"):
        compare(got, want, stats=False, label="rate", log=False)
    clean = _want(R, k)
    big = {key: np.concatenate([v, clean[key]]) for key, v in want.items()}   # 160,000 rows: one may be exempt
    gbig = {key: np.concatenate([v, clean[key]]) for key, v in got.items()}
    assert compare(gbig, big, stats=False, label="rate ok", log=False) == 1


def test_threaded_oracle_equals_one_call():
    """The GPU tests run the oracle on request ranges in host threads; the concatenated outputs
    equal one call over the whole batch, bit for bit."""
    import torch

    import oracle
    import workloads
    from tests.sampling_parity import by_request

    w = workloads.sample_batch(37, 3, 3000, 700, torch.bfloat16, T=[(0.7, 0.0, 1.1)[r % 3] for r in range(37)],
                               sigma_pos=0.8, delta=2.0,
                               seed=3, device="cpu")
    R, k = w["R"], w["k"]
    t, d = workloads.host_rows(w["target"]), workloads.host_rows(w["draft_logits"])
    d2t, draft = w["d2t"].numpy(), w["draft"].numpy()
    seeds, T = w["seeds"].numpy().view(np.uint64), w["temperature"].numpy()
    one = oracle.verify_sample(t, d, d2t, R, k, draft, seeds, T)
    par = by_request(lambda lo, hi: oracle.verify_sample(t[lo * (k + 1):hi * (k + 1)], d[lo * k:hi * k], d2t,
                                                         hi - lo, k, draft[lo:hi], seeds[lo:hi], T[lo:hi]), R,
                     threads=4)
    assert set(one) == set(par)
    for key in one:
        np.testing.assert_array_equal(np.nan_to_num(one[key]), np.nan_to_num(par[key]), err_msg=key)
