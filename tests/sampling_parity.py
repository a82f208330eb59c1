"""Comparison of the CUDA sampling outputs with the oracle's (test helper).

Tokens, accept lengths and status must be identical except for requests with
a row whose decision margin is below 1e-6 (|u - p/q| of a tested position, or
the relative gap between the two smallest race keys of the row the race ran
on), measured by the oracle in fp64.  Those rows are exempt: they are counted
per row (a CFG codebook row counts on its own), and every comparison requires
fewer than 1e-5 of its rows to be exempt, which for fewer than 10^5 rows
means none.  The counts are logged and printed at the end of the session.
p(x_j) and q(x_j) must agree within 1e-5 relative (absolute floor 1e-9, for
values near fp32 underflow).  TV must agree within 1e-5 relative or 1e-6
absolute: the kernel evaluates every probability in fp32 with ~1e-6 relative
error (rounding of c = log2(e)/T times the logit spread, ex2.approx's 2 ulp,
the normaliser's sum), so a sum of |p - q| carries an absolute error of that
order however small TV is.
"""
from __future__ import annotations

import os

import numpy as np

from oracle import MARGIN, exempt_rows  # noqa: F401  (the rule lives beside the oracle's margins)

EXEMPT_RATE = 1e-5  # exempt rows must be fewer than this share of the rows compared
REL = 1e-5
EXEMPT_LOG = []  # (label, exempt rows, rows compared) of every comparison of the session
ABS_FLOOR = {"tv": 1e-6, "p_draft": 1e-9, "q_draft": 1e-9}


def close(got, want, name=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), "NaN pattern differs"
    g, w = got[~nan_w], want[~nan_w]
    tol = np.maximum(REL * np.abs(w), ABS_FLOOR.get(name, 1e-9))
    bad = np.abs(g - w) > tol
    if bad.any():
        i = np.argmax(np.abs(g - w) - tol)
        raise AssertionError(f"{name}: {bad.sum()} values off; worst got {g[i]:.9g} want {w[i]:.9g} "
                             f"(rel {abs(g[i] - w[i]) / max(abs(w[i]), 1e-300):.3g}) at flat index {i}")


def commits_at_least_one_token(accept_len, tokens):
    """The pass-level invariant of the pages: every pass commits its n accepted drafts and
    one more token (n + 1 >= 1 valid ids per request, frames of S ids for CFG), so a
    speculative pass never does worse than one autoregressive step; -1 after them."""
    R = len(accept_len)
    t = np.asarray(tokens).reshape(R, -1)
    k1 = t.shape[1]
    n = np.asarray(accept_len)
    per = 1
    if tokens.ndim == 3:  # [R, k + 1, S]
        k1, per = tokens.shape[1], tokens.shape[2]
    assert np.all((n >= 0) & (n <= k1 - 1)), "accept length outside [0, k]"
    idx = np.arange(k1 * per)[None, :] // per
    committed = idx <= n[:, None]
    assert np.all(t[committed] >= 0), "a committed token is not a vocabulary id"
    assert np.all(t[~committed] == -1), "padding after the committed tokens is not -1"


def compare(got: dict, want: dict, stats=True, label=None, log=True, pooled=False):
    """got: CUDA outputs (numpy); want: oracle outputs.  Checks the parity rule and, unless the
    caller pools several comparisons (then it asserts the pooled rate), the exempt-row rate;
    returns the number of exempt rows."""
    commits_at_least_one_token(got["accept_len"], got["tokens"])
    commits_at_least_one_token(want["accept_len"], want["tokens"])
    rows_ex = exempt_rows(want)
    exempt_req = rows_ex.any(axis=1)
    R = len(want["accept_len"])
    same = (got["accept_len"] == want["accept_len"]) & np.all(
        got["tokens"].reshape(R, -1) == want["tokens"].reshape(R, -1), axis=1)
    if "status" in got:
        same &= got["status"] == want["status"]
    bad = ~same & ~exempt_req
    assert not bad.any(), (f"{bad.sum()} non-exempt requests differ, e.g. request {np.nonzero(bad)[0][:5]}: "
                           f"got {got['accept_len'][bad][:5]} {got['tokens'].reshape(R, -1)[bad][:2]} want "
                           f"{want['accept_len'][bad][:5]} {want['tokens'].reshape(R, -1)[bad][:2]}")
    if stats:
        for key in ("tv", "p_draft", "q_draft"):
            if key in got and key in want:
                close(got[key], want[key], key)
    n_ex, n_rows = int(rows_ex.sum()), int(rows_ex.size)
    if label is None:
        label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    if log:
        EXEMPT_LOG.append((label, n_ex, n_rows, int((~same).sum())))
    if not pooled:
        assert n_ex < EXEMPT_RATE * n_rows, f"{n_ex} exempt rows of {n_rows}: not below {EXEMPT_RATE:g} of the rows"
    return n_ex


def assert_pooled_rate(exempt: int, rows: int):
    """The rate rule over comparisons pooled until they hold at least 1 / EXEMPT_RATE rows."""
    assert rows * EXEMPT_RATE >= 1, f"only {rows} rows pooled"
    assert exempt < EXEMPT_RATE * rows, f"{exempt} exempt rows of {rows}: not below {EXEMPT_RATE:g} of the rows"


def oracle_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def by_request(fn, R: int, threads: int | None = None):
    """fn(lo, hi) -> the oracle's outputs for requests [lo, hi).  The ranges run on host threads
    (the oracle is C called through ctypes, which releases the GIL; every call owns its
    buffers) and the outputs are concatenated in request order."""
    import concurrent.futures as cf

    threads = threads or oracle_threads()
    per = max(1, -(-R // (4 * threads)))
    spans = [(lo, min(R, lo + per)) for lo in range(0, R, per)]
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        outs = list(ex.map(lambda sp: fn(*sp), spans))
    return {key: np.concatenate([o[key] for o in outs]) for key in outs[0]}
