"""Pins of the fp64 CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print for the worked example, known-answer vectors of Philox4x32-10,
closed forms, identities between two different outputs of the oracle,
brute-force autoregressive decoding and chi-square tests of the sampled
distribution.  None of them needs a GPU.
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle
from tests.conftest import golden

CHI2_ALPHA = 1e-3


def _chi2_ok(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    keep = probs > 0
    assert counts[~keep].sum() == 0, "mass where the target probability is 0"
    exp = probs[keep] / probs[keep].sum() * counts.sum()
    return stats.chisquare(counts[keep], exp).pvalue


# --------------------------------------------------------------------------
# Philox4x32-10 and the uniform
# --------------------------------------------------------------------------
def test_philox_known_answers():
    for v in golden("philox_kat.json")["vectors"]:
        ctr = [int(h, 16) for h in v["ctr"]]
        key = [int(h, 16) for h in v["key"]]
        out = [int(h, 16) for h in v["out"]]
        assert list(oracle.philox4x32_10(ctr, key)) == out


def test_uniform_open_interval_and_exact_in_fp32():
    assert oracle.uniform_from_word(0) == 2.0 ** -24
    assert oracle.uniform_from_word(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    rng = np.random.default_rng(1)
    for r in rng.integers(0, 2 ** 32, size=2000, dtype=np.uint64):
        u = oracle.uniform_from_word(int(r))
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u  # both sides see the same u


def test_uniform_counter_layout():
    # element x of (seed, row, tag) is word x & 3 of Philox((x>>2, row, tag, 0), seed)
    seed = 0x0123456789ABCDEF
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for x, row, tag in [(0, 0, 0), (5, 3, 1), (151935, 8, 2), (7, 31, 1)]:
        words = oracle.philox4x32_10([x >> 2, row, tag, 0], key)
        assert oracle.uniform(seed, row, tag, x) == oracle.uniform_from_word(int(words[x & 3]))


# --------------------------------------------------------------------------
# the exponential race samples w / sum(w)
# --------------------------------------------------------------------------
def test_race_single_support_and_zero_weights():
    w = np.zeros(9)
    w[6] = 1e-30
    for seed in range(50):
        assert oracle.race(w, seed, 0, 1)[0] == 6
    assert oracle.race(np.zeros(4), 3, 0, 1)[0] == -1


def test_race_distribution_chi_square():
    w = np.array([0.05, 0.0, 0.4, 0.15, 0.3, 0.1])
    n = 100_000
    counts = np.zeros(len(w))
    for seed in range(n):
        counts[oracle.race(w, seed * 7919 + 11, 2, 2)[0]] += 1
    assert _chi2_ok(counts, w) > CHI2_ALPHA


def test_race_distribution_ragged_row_with_zeros():
    # 23 ids (not a multiple of the four uniforms a Philox block gives), zeros inside
    rng = np.random.default_rng(5)
    w = rng.uniform(0.0, 1.0, 23) ** 3
    w[[1, 9, 10, 22]] = 0.0
    n = 60_000
    counts = np.zeros(len(w))
    for seed in range(n):
        counts[oracle.race(w, seed * 104729 + 3, 5, 1)[0]] += 1
    assert _chi2_ok(counts, w) > CHI2_ALPHA


def test_race_counter_layout_and_margin():
    # the uniform of a candidate is counted by its absolute id x (block x >> 2, word x & 3), the
    # row and the tag; the margin is the relative gap between the two smallest keys
    V = 151_936
    ids = np.array([4100, 4101, 4102, 77_777, V - 1])
    w = np.zeros(V)
    w[ids] = [0.2, 0.5, 0.3, 0.25, 0.4]
    for seed in range(40):
        keys = np.array([-math.log(oracle.uniform(seed, 9, 1, int(x))) / w[x] for x in ids])
        got, margin = oracle.race(w, seed, 9, 1)
        assert got == ids[int(np.argmin(keys))]
        ks = np.sort(keys)
        assert margin == pytest.approx((ks[1] - ks[0]) / ks[0], rel=1e-12)
    # another row or tag draws other uniforms, so the winners differ for some seeds
    same_row = [oracle.race(w, s, 9, 1)[0] for s in range(40)]
    assert same_row != [oracle.race(w, s, 8, 1)[0] for s in range(40)]
    assert same_row != [oracle.race(w, s, 9, 2)[0] for s in range(40)]


# --------------------------------------------------------------------------
# worked example of the blog (p = [.5,.3,.2], q = [.4,.4,.2])
# --------------------------------------------------------------------------
def _example_inputs(R, draft_tokens):
    g = golden("worked_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    target = np.tile(np.log(p).astype(np.float32), (2 * R, 1))  # rows: position 0, bonus
    draft_logits = np.tile(np.log(q).astype(np.float32), (R, 1))
    draft = np.asarray(draft_tokens, np.int32).reshape(R, 1)
    return g, p, q, target, draft_logits, draft


def test_worked_example_statistics():
    g, p, q, target, dl, draft = _example_inputs(3, [0, 1, 2])
    out = oracle.verify_sample(target, dl, None, 3, 1, draft, np.arange(3), np.ones(3))
    assert np.allclose(out["tv"][:, 0], g["tv"], atol=1e-7)
    assert np.allclose(out["p_draft"][:, 0], p, atol=1e-7)
    assert np.allclose(out["q_draft"][:, 0], q, atol=1e-7)
    assert out["p_draft"][1, 0] / out["q_draft"][1, 0] == pytest.approx(g["accept_prob_of_draft"], abs=1e-7)
    assert 1.0 - out["tv"][0, 0] == pytest.approx(g["alpha"], abs=1e-7)


def test_worked_example_output_distribution():
    R = 1_000_000
    rng = np.random.default_rng(2024)
    g, p, q, *_ = _example_inputs(1, [0])
    x = rng.choice(3, size=R, p=q)
    _, _, _, target, dl, draft = _example_inputs(R, x)
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.verify_sample(target, dl, None, R, 1, draft, seeds, np.ones(R, np.float32))
    first = out["tokens"][:, 0]
    counts = np.bincount(first, minlength=3)
    assert _chi2_ok(counts, g["output_distribution"]) > CHI2_ALPHA
    accepted = out["accept_len"] == 1
    # overall acceptance = 1 - TV; B is accepted with p(B)/q(B) = 0.75
    assert abs(accepted.mean() - g["alpha"]) < 5 * math.sqrt(0.09 / R)
    isB = x == 1
    assert abs(accepted[isB].mean() - g["accept_prob_of_draft"]) < 5 * math.sqrt(0.1875 / isB.sum())
    # residual normalised is [1, 0, 0]: rejections emit A (up to the fp32 rounding of ln p, ln q)
    assert np.mean(first[~accepted] != 0) < 1e-4
    # after acceptance the bonus comes from p (row 1)
    assert _chi2_ok(np.bincount(out["tokens"][accepted, 1], minlength=3), p) > CHI2_ALPHA


# --------------------------------------------------------------------------
# alpha = 1 - TV and sum max(0, p - q) = TV, from two different oracle paths
# --------------------------------------------------------------------------
def _all_draft_tokens(target_row, draft_row, d2t, V, T=1.0):
    """One request per target id x with draft token x: p(x), q(x) and TV."""
    R = V
    target = np.tile(target_row, (2 * R, 1))
    dl = np.tile(draft_row, (R, 1))
    out = oracle.verify_sample(target, dl, d2t, R, 1, np.arange(V, dtype=np.int32).reshape(R, 1),
                               np.arange(R), np.full(R, T, np.float32))
    return out["p_draft"][:, 0], out["q_draft"][:, 0], out["tv"][:, 0], out


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_alpha_equals_one_minus_tv(T):
    rng = np.random.default_rng(int(T * 10))
    V = 64
    z = rng.normal(0, 2, V).astype(np.float32)
    y = (z + rng.normal(0, 1, V)).astype(np.float32)
    p, q, tv, _ = _all_draft_tokens(z, y, None, V, T)
    assert np.allclose(tv, tv[0], rtol=0, atol=0)  # TV does not depend on the draft token
    assert p.sum() == pytest.approx(1.0, abs=1e-12)
    assert q.sum() == pytest.approx(1.0, abs=1e-12)
    alpha = np.sum(q * np.minimum(1.0, p / q))
    assert alpha == pytest.approx(1.0 - tv[0], abs=1e-12)
    assert np.sum(np.maximum(0.0, p - q)) == pytest.approx(tv[0], abs=1e-12)


def test_infinite_and_tiny_temperatures_closed_forms():
    # T = +inf: p uniform over the V target ids and q over the Vd support ids, so
    # TV = 1 - Vd / V, every on-support draft has p/q = Vd / V and every off-support one is
    # rejected.  T -> 0: p and q one-hot at their argmaxes, TV 0 or 1.
    rng = np.random.default_rng(21)
    V, Vd = 40, 12
    d2t = rng.permutation(V)[:Vd].astype(np.int32)
    z = rng.normal(0, 1.5, V).astype(np.float32)
    y = (z[d2t] + rng.normal(0, 0.5, Vd)).astype(np.float32)
    p, q, tv, out = _all_draft_tokens(z, y, d2t, V, T=np.inf)
    assert np.allclose(p, 1.0 / V, rtol=1e-12)
    assert np.allclose(q[d2t], 1.0 / Vd, rtol=1e-12) and np.all(np.delete(q, d2t) == 0)
    assert np.allclose(tv, 1.0 - Vd / V, atol=1e-12)
    p, q, tv, out = _all_draft_tokens(z, y, d2t, V, T=1e-6)
    zmax, ymax = int(np.argmax(z)), int(d2t[np.argmax(y)])
    assert p[zmax] == 1.0 and np.all(np.delete(p, zmax) == 0.0)
    assert q[ymax] == 1.0 and np.all(np.delete(q, ymax) == 0.0)
    assert np.all(tv == (0.0 if zmax == ymax else 1.0))


def test_truncated_vocabulary_tv_over_full_support():
    rng = np.random.default_rng(5)
    V, Vd = 40, 12
    d2t = rng.permutation(V)[:Vd].astype(np.int32)
    z = rng.normal(0, 1.5, V).astype(np.float32)
    y = (z[d2t] + rng.normal(0, 0.5, Vd)).astype(np.float32)
    p, q, tv, out = _all_draft_tokens(z, y, d2t, V)
    off = np.setdiff1d(np.arange(V), d2t)
    assert np.all(q[off] == 0.0)
    assert q.sum() == pytest.approx(1.0, abs=1e-12)
    # off-support drafts are always rejected and flagged
    assert np.all(out["accept_len"][off] == 0)
    assert np.all(out["status"][off] & oracle.ST_OFF_SUPPORT)
    # TV over the full target vocabulary: 1 - sum min(p, q), which includes p's off-support mass
    assert tv[0] == pytest.approx(1.0 - np.minimum(p, q).sum(), abs=1e-12)
    tv_support_only = 0.5 * np.abs(p[d2t] / p[d2t].sum() - q[d2t]).sum()
    assert abs(tv_support_only - tv[0]) > 1e-3  # the mismatch the blog warns about


# --------------------------------------------------------------------------
# chi-square: output = p, residual branch = norm(max(0, p - q)), bonus = p
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V,T", [(5, 1.0), (8, 0.6)])
def test_sampling_output_distribution_chi_square(V, T):
    R = 1_000_000
    rng = np.random.default_rng(V)
    z0 = rng.normal(0, 1.2, V).astype(np.float32)
    zb = rng.normal(0, 1.2, V).astype(np.float32)
    y0 = rng.normal(0, 1.2, V).astype(np.float32)
    p = np.exp(z0.astype(np.float64) / T); p /= p.sum()
    pb = np.exp(zb.astype(np.float64) / T); pb /= pb.sum()
    q = np.exp(y0.astype(np.float64) / T); q /= q.sum()
    x = rng.choice(V, size=R, p=q)
    target = np.empty((2 * R, V), np.float32)
    target[0::2] = z0
    target[1::2] = zb
    dl = np.tile(y0, (R, 1))
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.verify_sample(target, dl, None, R, 1, x.reshape(R, 1).astype(np.int32), seeds,
                               np.full(R, T, np.float32))
    first = out["tokens"][:, 0]
    acc = out["accept_len"] == 1
    assert _chi2_ok(np.bincount(first, minlength=V), p) > CHI2_ALPHA
    resid = np.maximum(0.0, p - q)
    assert _chi2_ok(np.bincount(first[~acc], minlength=V), resid) > CHI2_ALPHA
    assert _chi2_ok(np.bincount(out["tokens"][acc, 1], minlength=V), pb) > CHI2_ALPHA
    tv = 0.5 * np.abs(p - q).sum()
    assert abs(acc.mean() - (1 - tv)) < 5 * math.sqrt(tv * (1 - tv) / R)


def _binned(tokens, probs, heavy, chunk):
    """counts and probabilities over bins: each heavy id alone, then the rest of each chunk"""
    V = probs.size
    bin_of = np.arange(V) // chunk + len(heavy)
    bin_of[heavy] = np.arange(len(heavy))
    nb = len(heavy) + (V + chunk - 1) // chunk
    return np.bincount(bin_of[tokens], minlength=nb), np.bincount(bin_of, weights=probs, minlength=nb)


TAIL_BIN = 2048  # ids per bin of the long tail in the binned chi-square tests


def test_sampling_distribution_long_row():
    # a row of 4100 ids with mass on a few ids far apart and on the long tail (binned in 2048s)
    V, T, R = 2 * TAIL_BIN + 4, 1.0, 8_000
    rng = np.random.default_rng(11)
    heavy = np.array([3, 2050, 4099])
    z0 = rng.normal(0, 0.5, V).astype(np.float32)
    zb = rng.normal(0, 0.5, V).astype(np.float32)
    y0 = rng.normal(0, 0.5, V).astype(np.float32)
    z0[heavy] = [7.0, 6.0, 7.5]
    zb[heavy] = [6.5, 7.5, 6.0]
    y0[[3, 1000, 3000]] = [8.0, 7.0, 6.0]
    p = np.exp(z0.astype(np.float64) / T); p /= p.sum()
    pb = np.exp(zb.astype(np.float64) / T); pb /= pb.sum()
    q = np.exp(y0.astype(np.float64) / T); q /= q.sum()
    x = rng.choice(V, size=R, p=q)
    target = np.empty((2 * R, V), np.float32)
    target[0::2] = z0
    target[1::2] = zb
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.verify_sample(target, np.tile(y0, (R, 1)), None, R, 1, x.reshape(R, 1).astype(np.int32),
                               seeds, np.full(R, T, np.float32))
    first = out["tokens"][:, 0]
    acc = out["accept_len"] == 1
    assert _chi2_ok(*_binned(first, p, heavy, TAIL_BIN)) > CHI2_ALPHA
    resid = np.maximum(0.0, p - q)
    assert _chi2_ok(*_binned(first[~acc], resid, heavy, TAIL_BIN)) > CHI2_ALPHA
    assert _chi2_ok(*_binned(out["tokens"][acc, 1], pb, heavy, TAIL_BIN)) > CHI2_ALPHA


def test_tokens_per_pass_closed_form():
    """i.i.d. positions with a fixed (p, q): E[tokens] = (1 - a^(k+1)) / (1 - a)."""
    R, k, V = 400_000, 4, 6
    rng = np.random.default_rng(77)
    z = rng.normal(0, 1, V).astype(np.float32)
    y = rng.normal(0, 1, V).astype(np.float32)
    p = np.exp(z.astype(np.float64)); p /= p.sum()
    q = np.exp(y.astype(np.float64)); q /= q.sum()
    a = 1 - 0.5 * np.abs(p - q).sum()
    target = np.tile(z, (R * (k + 1), 1))
    dl = np.tile(y, (R * k, 1))
    x = rng.choice(V, size=(R, k), p=q).astype(np.int32)
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.verify_sample(target, dl, None, R, k, x, seeds, np.ones(R, np.float32))
    tokens = out["accept_len"] + 1
    expect = (1 - a ** (k + 1)) / (1 - a)
    assert abs(tokens.mean() - expect) < 5 * tokens.std() / math.sqrt(R)
    assert np.all(tokens >= 1)


def test_dspark_arithmetic():
    g = golden("dspark_metrics.json")
    acc = np.array(g["per_position_accept"])
    assert np.cumprod(acc).sum() == pytest.approx(g["independence_accept_len"], abs=5e-3)
    a = g["equivalent_constant_alpha"]
    k = len(acc)
    assert sum(a ** i for i in range(1, k + 1)) == pytest.approx(g["reported_accept_len"], abs=5e-3)
    assert (1 - a ** (k + 1)) / (1 - a) == pytest.approx(g["tokens_per_pass"], abs=5e-3)
    for c, s in zip(g["draft_cost"], g["net_speedup"]):
        assert g["tokens_per_pass"] / (1 + k * c) == pytest.approx(s, abs=5e-3)
    assert 1 - g["raw_tv"] == pytest.approx(g["accept_rate_epoch"], abs=1e-9)


# --------------------------------------------------------------------------
# sampling is lossless end to end: two emitted tokens ~ p(s1) p(s2 | s1)
# --------------------------------------------------------------------------
def _toy_logits(ctx, V, scale=1.0, salt=0):
    h = abs(hash((salt,) + tuple(int(c) for c in ctx))) % (2 ** 32)
    return (np.random.default_rng(h).normal(0, scale, V)).astype(np.float32)


def test_sampling_stream_convention():
    """Which uniforms decide: position j's accept test takes element 0 of (row j, tag 0); the
    residual race at the first rejection n takes (row n, tag 1); the bonus race (row k, tag 2).
    The expected tokens are rebuilt here from p and q in numpy and the library-independent
    race/uniform pins above, so a swapped tag or row in the verify path fails."""
    V, k, T, R = 6, 2, 0.8, 300
    rng = np.random.default_rng(31)
    z = rng.normal(0, 1.0, (R * (k + 1), V)).astype(np.float32)
    y = rng.normal(0, 1.0, (R * k, V)).astype(np.float32)
    draft = rng.integers(0, V, size=(R, k)).astype(np.int32)
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.verify_sample(z, y, None, R, k, draft, seeds, np.full(R, T, np.float32))

    def sm(v):
        e = np.exp(v.astype(np.float64) / T - (v.astype(np.float64) / T).max())
        return e / e.sum()

    for r in range(R):
        sd = int(seeds[r])
        n = k
        for j in range(k):
            p, q = sm(z[r * (k + 1) + j]), sm(y[r * k + j])
            x = draft[r, j]
            if not oracle.uniform(sd, j, 0, 0) < p[x] / q[x]:
                n = j
                want = oracle.race(np.maximum(p - q, 0.0), sd, j, 1)[0]
                break
        if n == k:
            want = oracle.race(sm(z[r * (k + 1) + k]), sd, k, 2)[0]
        assert out["accept_len"][r] == n
        assert out["tokens"][r, n] == want


def test_sampling_matches_autoregressive_pairs():
    V, T, n = 3, 1.0, 300_000
    rng = np.random.default_rng(9)
    ctx0 = (1, 2)

    def p_of(ctx):
        z = _toy_logits(ctx, V, 1.3).astype(np.float64) / T
        e = np.exp(z - z.max())
        return e / e.sum()

    def q_of(ctx):
        z = _toy_logits(ctx, V, 1.3, salt=1).astype(np.float64) / T
        e = np.exp(z - z.max())
        return e / e.sum()

    # one verify call with k = 1 per trial, then a second call when only one token came out
    qs0 = q_of(ctx0)
    drafts = rng.choice(V, size=n, p=qs0).astype(np.int32)
    target = np.empty((2 * n, V), np.float32)
    target[0::2] = _toy_logits(ctx0, V, 1.3)
    for v in range(V):
        target[1::2][drafts == v] = _toy_logits(ctx0 + (v,), V, 1.3)
    dl = np.tile(_toy_logits(ctx0, V, 1.3, salt=1), (n, 1))
    seeds = rng.integers(0, 2 ** 63, size=n, dtype=np.uint64)
    out = oracle.verify_sample(target, dl, None, n, 1, drafts.reshape(n, 1), seeds, np.full(n, T, np.float32))
    s1 = out["tokens"][:, 0]
    s2 = out["tokens"][:, 1].copy()
    need = out["accept_len"] == 0
    # a second call from context ctx0 + (s1,) supplies s2 for the short ones
    idx = np.nonzero(need)[0]
    m = len(idx)
    target2 = np.empty((2 * m, V), np.float32)
    dl2 = np.empty((m, V), np.float32)
    drafts2 = np.empty(m, np.int32)
    for v in range(V):
        sel = s1[idx] == v
        ctx = ctx0 + (v,)
        target2[0::2][sel] = _toy_logits(ctx, V, 1.3)
        dl2[sel] = _toy_logits(ctx, V, 1.3, salt=1)
        drafts2[sel] = rng.choice(V, size=sel.sum(), p=q_of(ctx))
    for v in range(V):
        for w in range(V):
            sel = (s1[idx] == v) & (drafts2 == w)
            target2[1::2][sel] = _toy_logits(ctx0 + (v, w), V, 1.3)
    seeds2 = rng.integers(0, 2 ** 63, size=m, dtype=np.uint64)
    out2 = oracle.verify_sample(target2, dl2, None, m, 1, drafts2.reshape(m, 1), seeds2, np.full(m, T, np.float32))
    s2[idx] = out2["tokens"][:, 0]
    joint = np.zeros(V * V)
    np.add.at(joint, s1 * V + s2, 1)
    p1 = p_of(ctx0)
    expect = np.array([p1[a] * p_of(ctx0 + (a,))[b] for a in range(V) for b in range(V)])
    assert _chi2_ok(joint, expect) > CHI2_ALPHA


# --------------------------------------------------------------------------
# greedy verification reproduces autoregressive argmax decoding
# --------------------------------------------------------------------------
def _ar_greedy(ctx, L, V):
    out = []
    for _ in range(L):
        t = int(np.argmax(_toy_logits(tuple(ctx) + tuple(out), V)))
        out.append(t)
    return out


@pytest.mark.parametrize("branches", [1, 2, 4])
def test_greedy_verification_equals_autoregressive(branches):
    V, k, L = 50, 6, 120
    rng = np.random.default_rng(branches)
    ctx = (3, 1, 4)
    ar = _ar_greedy(ctx, L, V)
    out = []
    calls = 0
    while len(out) < L:
        base = tuple(ctx) + tuple(out)
        # main draft: the model's own greedy continuation, each token corrupted w.p. 0.3
        main = []
        for _ in range(k):
            t = int(np.argmax(_toy_logits(base + tuple(main), V)))
            if rng.random() < 0.3:
                t = int(rng.integers(0, V))
            main.append(t)
        rows = [_toy_logits(base + tuple(main[:j]), V) for j in range(k + 1)]
        drafts = [main]
        # further branches (a tree of first tokens): the best ids of row 0 other than the main
        # draft's first token, each continued greedily
        row0 = rows[0].astype(np.float64)
        firsts = [int(t) for t in np.argsort(-row0, kind="stable") if int(t) != main[0]][:branches - 1]
        for first in firsts:
            runner = [first]
            for _ in range(k - 1):
                runner.append(int(np.argmax(_toy_logits(base + tuple(runner), V))))
            rows += [_toy_logits(base + tuple(runner[:j]), V) for j in range(1, k + 1)]
            drafts.append(runner)
        res = oracle.verify_greedy(np.stack(rows), 1, k, branches, np.array(drafts, np.int32))
        n = int(res["accept_len"][0])
        committed = res["tokens"][0, : n + 1].tolist()
        assert len(committed) >= 1 and all(t >= 0 for t in committed)
        assert np.all(res["tokens"][0, n + 1:] == -1)
        out.extend(committed)
        calls += 1
    assert out[:L] == ar
    assert calls < L  # drafts were actually accepted


def test_greedy_branch_selection_rules():
    V, k = 8, 3

    def rows_with_argmax(ams):
        r = np.zeros((len(ams), V), np.float32)
        for i, a in enumerate(ams):
            r[i, a] = 5.0
        return r

    # rows: [p1 | main p2..p4 | runner p2..p4]
    rows = rows_with_argmax([2, 3, 4, 5, 6, 7, 0])
    # both branches start with the argmax of row 0; main matches 1, runner matches 2 -> runner wins
    res = oracle.verify_greedy(rows, 1, k, 2, np.array([[2, 3, 0], [2, 6, 7]], np.int32))
    assert res["branch"][0] == 1 and res["accept_len"][0] == 3
    assert res["tokens"][0].tolist() == [2, 6, 7, 0]
    # equal n -> branch 0
    res = oracle.verify_greedy(rows, 1, k, 2, np.array([[2, 3, 1], [2, 6, 1]], np.int32))
    assert res["branch"][0] == 0 and res["accept_len"][0] == 2
    assert res["tokens"][0].tolist() == [2, 3, 4, -1]
    # only the runner is viable
    res = oracle.verify_greedy(rows, 1, k, 2, np.array([[1, 3, 4], [2, 6, 7]], np.int32))
    assert res["branch"][0] == 1 and res["accept_len"][0] == 3
    # none viable: n = 0, branch 0, correction = argmax of row 0
    res = oracle.verify_greedy(rows, 1, k, 2, np.array([[1, 3, 4], [0, 6, 7]], np.int32))
    assert res["branch"][0] == 0 and res["accept_len"][0] == 0
    assert res["tokens"][0].tolist() == [2, -1, -1, -1]


def test_tree_branch_selection_rules():
    """Four branches sharing row 0: the viable branch with the longest accepted prefix wins,
    ties go to the lowest branch; rows are [p1 | b0 p2..p4 | b1 .. | b2 .. | b3 ..]."""
    V, k, B = 10, 3, 4
    ams = [2, 3, 4, 5, 6, 7, 1, 8, 9, 0, 3, 4, 5]  # argmax of row 0, then three rows per branch
    rows = np.zeros((1 + B * k, V), np.float32)
    for i, a in enumerate(ams):
        rows[i, a] = 5.0
    # accepted prefixes 2, 3, 3 and a branch that is not viable: branch 1 (the first of the longest)
    drafts = np.array([[2, 3, 0], [2, 6, 7], [2, 8, 9], [1, 3, 4]], np.int32)
    res = oracle.verify_greedy(rows, 1, k, B, drafts)
    assert res["accept_len"][0] == 3 and res["branch"][0] == 1
    assert res["tokens"][0].tolist() == [2, 6, 7, 1]
    # accepted prefixes 2, 1, 1, 1: branch 0, its correction from its own row
    drafts = np.array([[2, 3, 0], [2, 5, 6], [2, 1, 8], [2, 0, 3]], np.int32)
    res = oracle.verify_greedy(rows, 1, k, B, drafts)
    assert res["accept_len"][0] == 2 and res["branch"][0] == 0
    assert res["tokens"][0].tolist() == [2, 3, 4, -1]
    # only the last branch is viable
    drafts = np.array([[1, 3, 4], [0, 6, 7], [9, 8, 9], [2, 3, 4]], np.int32)
    res = oracle.verify_greedy(rows, 1, k, B, drafts)
    assert res["accept_len"][0] == 3 and res["branch"][0] == 3
    assert res["tokens"][0].tolist() == [2, 3, 4, 5]


def test_greedy_ties_nan_inf_and_ranges():
    V = 6
    rows = np.zeros((3, V), np.float32)
    rows[0] = [1, 3, 3, 0, 3, 2]            # tie -> lowest index 1
    rows[1] = [np.nan, 0, 7, np.nan, 7, 1]  # NaN reads as -inf; tie -> 2
    rows[2] = [-np.inf] * V                  # all -inf -> index 0
    res = oracle.verify_greedy(rows, 1, 2, 1, np.array([[1, 2]], np.int32))
    assert res["accept_len"][0] == 2 and res["tokens"][0].tolist() == [1, 2, 0]
    assert res["status"][0] & oracle.ST_BAD_LOGITS
    res = oracle.verify_greedy(rows[:2], 1, 1, 1, np.array([[V + 3]], np.int32))
    assert res["accept_len"][0] == 0 and res["tokens"][0].tolist() == [1, -1]
    assert res["status"][0] & oracle.ST_TOKEN_RANGE
    # k = 0: one autoregressive step
    res = oracle.verify_greedy(rows[:1], 1, 0, 1, np.zeros((1, 0), np.int32))
    assert res["accept_len"][0] == 0 and res["tokens"][0].tolist() == [1]
    # +inf is a legal maximum for greedy but is flagged
    r = np.zeros((1, V), np.float32)
    r[0, 4] = np.inf
    res = oracle.verify_greedy(r, 1, 0, 1, np.zeros((1, 0), np.int32))
    assert res["tokens"][0].tolist() == [4] and res["status"][0] & oracle.ST_BAD_LOGITS


def _top2_by_sort(rows):
    """the first two ids of each row under a stable sort by value, descending (NaN as -inf)"""
    v = np.where(np.isnan(rows), -np.inf, rows.astype(np.float64))
    order = np.argsort(-v, axis=1, kind="stable")
    return order[:, :2]


def test_top2_matches_a_stable_sort():
    rng = np.random.default_rng(31)
    rows = rng.integers(-3, 4, (400, 37)).astype(np.float32)  # many ties
    rows[rng.random(rows.shape) < 0.05] = np.nan
    rows[rng.random(rows.shape) < 0.05] = -np.inf
    rows[::7, 5] = np.inf
    got = oracle.top2_rows(rows)
    assert np.array_equal(got, _top2_by_sort(rows))
    bits = (rng.normal(0, 2, (50, 300)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(oracle.top2_rows(bits), _top2_by_sort(widened))


def test_top2_special_cases_and_greedy_argmax():
    rows = np.array([[1, 3, 3, 0, 3, 2],                       # tied maximum: its first two ids
                     [np.nan, 0, 7, np.nan, 5, 1],             # NaN reads as -inf
                     [-np.inf] * 6,                            # all -inf: ids 0 and 1
                     [2, -np.inf, -np.inf, -np.inf, -np.inf, -np.inf]], np.float32)
    assert oracle.top2_rows(rows).tolist() == [[1, 2], [2, 4], [0, 1], [0, 1]]
    assert oracle.top2_rows(np.array([[4.0], [np.nan]], np.float32)).tolist() == [[0, -1], [0, -1]]
    # the first id is the argmax of greedy verification
    rng = np.random.default_rng(32)
    z = rng.normal(0, 1, (9, 50)).astype(np.float32)
    z[:, 10] = z[:, 20] = z.max(axis=1) + 1.0
    res = oracle.verify_greedy(z, 1, 8, 1, np.full((1, 8), -1, np.int32))
    assert res["tokens"][0, 0] == oracle.top2_rows(z)[0, 0] == 10


def test_modality_is_the_partition_of_the_unmasked_argmax():
    """Text part [0, 100), codebooks [100, 164), [164, 228), a gap [228, 240) in no partition."""
    rng = np.random.default_rng(33)
    V, starts = 240, np.array([0, 100, 164, 228], np.int32)
    rows = rng.normal(0, 1, (60, V)).astype(np.float32)
    planted = rng.integers(0, V, 60)
    rows[np.arange(60), planted] = 9.0
    rows[0, 99] = rows[0, 100] = 20.0          # tie across a boundary: the lower id, text
    rows[1, :] = np.nan                       # all NaN: argmax 0
    rows[2, 230] = 30.0                       # in the gap: no partition
    rows[3, 164] = rows[4, 100] = rows[5, 227] = 30.0  # the first and the last id of a partition
    out = oracle.infer_modality(rows, starts)
    amax = _top2_by_sort(rows)[:, 0]
    assert np.array_equal(out["amax"], amax)
    want = np.searchsorted(starts, amax, side="right") - 1
    want[amax >= starts[-1]] = -1
    assert np.array_equal(out["part"], want)
    ok = want >= 0
    assert np.array_equal(out["mask_lo"][ok], starts[want[ok]])
    assert np.array_equal(out["mask_hi"][ok], starts[want[ok] + 1])
    assert np.all(out["mask_lo"][~ok] == 0) and np.all(out["mask_hi"][~ok] == 0)
    assert out["part"][:6].tolist() == [0, 0, -1, 2, 1, 2]


def test_bf16_rows_are_widened_exactly():
    rng = np.random.default_rng(3)
    V = 33
    f = rng.normal(0, 3, (4, V)).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    draft = np.array([[int(np.argmax(widened[0])), int(np.argmax(widened[1])), 0]], np.int32)
    a = oracle.verify_greedy(bits, 1, 3, 1, draft)
    b = oracle.verify_greedy(widened, 1, 3, 1, draft)
    assert a["tokens"].tolist() == b["tokens"].tolist()


def test_sampling_greedy_fallbacks():
    V, k = 5, 2
    rng = np.random.default_rng(4)
    z = rng.normal(0, 1, (k + 1, V)).astype(np.float32)
    y = rng.normal(0, 1, (k, V)).astype(np.float32)
    am = np.argmax(z, axis=1)
    draft = np.array([[am[0], (am[1] + 1) % V]], np.int32)
    for T, flag in [(0.0, 0), (-1.0, oracle.ST_BAD_TEMP), (np.nan, oracle.ST_BAD_TEMP)]:
        out = oracle.verify_sample(z, y, None, 1, k, draft, [7], [T])
        assert out["accept_len"][0] == 1 and out["tokens"][0].tolist() == [am[0], am[1], -1]
        assert out["status"][0] & oracle.ST_BAD_TEMP == flag
        assert np.all(np.isnan(out["tv"]))
    zb = z.copy()
    zb[2, 1] = np.nan
    out = oracle.verify_sample(zb, y, None, 1, k, draft, [7], [1.0])
    assert out["status"][0] & oracle.ST_BAD_LOGITS and out["tokens"][0].tolist() == [am[0], am[1], -1]


def test_accept_scan_brute_force():
    rng = np.random.default_rng(12)
    R, k = 500, 7
    acc = (rng.random((R, k)) < 0.8).astype(np.uint8)
    draft = rng.integers(0, 1000, (R, k)).astype(np.int32)
    fix = rng.integers(0, 1000, (R, k + 1)).astype(np.int32)
    out = oracle.accept_scan(acc, draft, fix)
    for r in range(R):
        n = 0
        while n < k and acc[r, n]:
            n += 1
        assert out["accept_len"][r] == n
        assert out["tokens"][r].tolist() == draft[r, :n].tolist() + [fix[r, n]] + [-1] * (k - n)


# --------------------------------------------------------------------------
# CFG merge: special weights reduce to plain verification
# --------------------------------------------------------------------------
def test_cfg_weight_zero_is_plain_sampling_of_uncond():
    rng = np.random.default_rng(21)
    R, k, W = 200, 3, 16
    c = rng.normal(0, 1, (R * (k + 1), W)).astype(np.float32)
    u = rng.normal(0, 1, (R * (k + 1), W)).astype(np.float32)
    y = (u[np.arange(R * (k + 1)) % (k + 1) != k] + rng.normal(0, 0.7, (R * k, W))).astype(np.float32)
    draft = rng.integers(0, W, (R, k)).astype(np.int32)
    seeds = rng.integers(0, 2 ** 63, R, dtype=np.uint64)
    T = np.full(R, 0.8, np.float32)
    a = oracle.cfg_merge_sample(c, u, [0], [0], 1, W, 0.0, y, R, k, draft, seeds, T)
    b = oracle.verify_sample(u, y, None, R, k, draft, seeds, T)
    assert np.array_equal(a["accept_len"], b["accept_len"])
    assert np.array_equal(a["tokens"][:, :, 0], b["tokens"])
    assert np.allclose(a["tv"][:, :, 0], b["tv"], atol=1e-15)


def test_cfg_without_drafts_draws_the_bonus_like_sampling():
    """k = 0: no draft rows, so the bonus follows the temperature alone, whether the draft
    logits are absent or empty.  With w = 0 (merged = u) and one codebook it is the sampling
    path's bonus on u: the same race, counter row 0, tag 2 (speculative decoding for Omni
    models, section 2: the bonus token is drawn from p)."""
    rng = np.random.default_rng(23)
    R, W = 300, 24
    c = rng.normal(0, 1, (R, W)).astype(np.float32)
    u = rng.normal(0, 1.5, (R, W)).astype(np.float32)
    seeds = rng.integers(0, 2 ** 63, R, dtype=np.uint64)
    T = np.where(np.arange(R) % 4 == 0, 0.0, 0.9).astype(np.float32)
    empty = np.zeros((R, 0), np.int32)
    a = oracle.cfg_merge_sample(c, u, [0], [0], 1, W, 0.0, None, R, 0, empty, seeds, T)
    a2 = oracle.cfg_merge_sample(c, u, [0], [0], 1, W, 0.0, np.zeros((0, W), np.float32), R, 0, empty, seeds, T)
    b = oracle.verify_sample(u, np.zeros((0, W), np.float32), None, R, 0, empty, seeds, T)
    assert np.array_equal(a["tokens"], a2["tokens"])
    assert np.array_equal(a["tokens"][:, :, 0], b["tokens"])
    sampled = T > 0
    assert np.all(a["tokens"][~sampled, 0, 0] == np.argmax(u[~sampled], axis=1))
    assert np.any(a["tokens"][sampled, 0, 0] != np.argmax(u[sampled], axis=1))  # drawn, not the argmax


def test_cfg_weight_one_greedy_is_greedy_on_cond():
    rng = np.random.default_rng(22)
    R, k, S, W = 30, 4, 3, 32
    f = rng.normal(0, 1, (2, R * (k + 1) * S, W)).astype(np.float32)
    c, u = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in f]  # bf16: c - u is exact here
    cw = (c.astype(np.uint32) << 16).view(np.float32)
    am = np.argmax(cw, axis=1).reshape(R, k + 1, S)
    base = np.array([1000 + W * s for s in range(S)], np.int32)
    draft = (am[:, :k, :] + base).astype(np.int32)
    draft[::3, 2, 1] = base[1] + (am[::3, 2, 1] + 1) % W  # some frames mismatch
    out = oracle.cfg_merge_sample(c, u, base, [0] * S, S, W, 1.0, None, R, k, draft,
                                  np.zeros(R, np.uint64), np.zeros(R, np.float32))
    for r in range(R):
        n = 2 if r % 3 == 0 else k
        assert out["accept_len"][r] == n
        assert out["tokens"][r, n].tolist() == (am[r, n] + base).tolist()


CFG_TAIL_BIN = 256  # ids per tail bin of the codebook-row chi-square test


def test_cfg_sampling_distribution_long_codebook_row():
    """A codebook row of 516 ids with mass on a few ids far apart and on the long tail: the
    emitted token follows p at the first frame, the residual where the draft was rejected,
    and p at the bonus frame."""
    W, T, R, w = 2 * CFG_TAIL_BIN + 4, 1.0, 8_000, 2.0
    rng = np.random.default_rng(24)
    heavy = np.array([3, 300, 513])
    cz = rng.normal(0, 0.3, W).astype(np.float32)
    uz = rng.normal(0, 0.3, W).astype(np.float32)
    cb = rng.normal(0, 0.3, W).astype(np.float32)
    cz[heavy] = [3.5, 3.0, 3.8]
    cb[heavy] = [3.2, 3.8, 3.0]
    yz = rng.normal(0, 0.5, W).astype(np.float32)
    yz[[3, 100, 400]] = [8.0, 7.0, 6.0]

    def merged(c):
        return (np.float32(w) * (c - uz) + uz).astype(np.float64)  # fp32 roundings, widened

    p = np.exp(merged(cz) / T); p /= p.sum()
    pb = np.exp(merged(cb) / T); pb /= pb.sum()
    q = np.exp(yz.astype(np.float64) / T); q /= q.sum()
    x = rng.choice(W, size=R, p=q)
    cond = np.empty((2 * R, W), np.float32)
    cond[0::2] = cz
    cond[1::2] = cb
    uncond = np.tile(uz, (2 * R, 1))
    seeds = rng.integers(0, 2 ** 63, size=R, dtype=np.uint64)
    out = oracle.cfg_merge_sample(cond, uncond, [0], [0], 1, W, w, np.tile(yz, (R, 1)), R, 1,
                                  x.reshape(R, 1, 1).astype(np.int32), seeds, np.full(R, T, np.float32))
    first = out["tokens"][:, 0, 0]
    acc = out["accept_len"] == 1
    assert _chi2_ok(*_binned(first, p, heavy, CFG_TAIL_BIN)) > CHI2_ALPHA
    resid = np.maximum(0.0, p - q)
    assert _chi2_ok(*_binned(first[~acc], resid, heavy, CFG_TAIL_BIN)) > CHI2_ALPHA
    assert _chi2_ok(*_binned(out["tokens"][acc, 1, 0], pb, heavy, CFG_TAIL_BIN)) > CHI2_ALPHA


def test_cfg_codebook_marginals_are_target():
    """Each codebook's emitted token at frame 0 follows its own p (S = 2)."""
    rng = np.random.default_rng(23)
    R, k, S, W = 300_000, 1, 2, 4
    cz = rng.normal(0, 1, (S, W)).astype(np.float32)
    uz = rng.normal(0, 1, (S, W)).astype(np.float32)
    yz = rng.normal(0, 1, (S, W)).astype(np.float32)
    w = 2.0
    cond = np.tile(np.concatenate([cz, cz]), (R, 1))   # frames 0 and 1 share logits
    uncond = np.tile(np.concatenate([uz, uz]), (R, 1))
    dl = np.tile(yz, (R, 1))
    merged = (uz.astype(np.float64) + w * (cz.astype(np.float64) - uz.astype(np.float64)))
    p = np.exp(merged - merged.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    q = np.exp(yz.astype(np.float64) - yz.max(1, keepdims=True)); q /= q.sum(1, keepdims=True)
    draft = np.stack([rng.choice(W, size=R, p=q[s]) for s in range(S)], axis=1).reshape(R, 1, S)
    seeds = rng.integers(0, 2 ** 63, R, dtype=np.uint64)
    out = oracle.cfg_merge_sample(cond, uncond, [0, 0], [0, 0], S, W, w, dl, R, k,
                                  draft.astype(np.int32), seeds, np.ones(R, np.float32))
    for s in range(S):
        assert _chi2_ok(np.bincount(out["tokens"][:, 0, s], minlength=W), p[s]) > CHI2_ALPHA


# --------------------------------------------------------------------------
# hypothesis pool ("Decode Before You Hear ...", method steps 3 and 5; the
# tool-call case study of Figure 6 (b))
# --------------------------------------------------------------------------
# token ids of the tool-call case study: "ok" (listen), "sure", "<call>", "find",
# "(", "TYO", ",", "Fri", ")", "</call>"
OK, SURE, CALL, FIND, LP, TYO, COMMA, FRI, RP, ENDCALL = 20, 21, 10, 11, 12, 13, 14, 15, 16, 17
CASE_DRAFTS = [
    [OK],                                             # chunk 1: listen
    [SURE, CALL, FIND, LP, TYO, COMMA, FRI, RP, ENDCALL],  # chunk 2: the call, drafted under silence
    [CALL, FIND, LP, TYO],                            # chunk 3: cut off by the window
    [OK],                                             # chunk 3: runner-up branch
]
CASE_POOL = [OK, -1, SURE, CALL, FIND, LP, TYO, COMMA, FRI, RP, ENDCALL, -1, CALL, FIND, LP, TYO, -1, OK, -1]


def _append_all(drafts, Lp, width=10):
    pool = np.full((1, Lp), -7, np.int32)  # contents beyond pool_len never matter
    plen = np.zeros(1, np.int32)
    statuses = []
    for d in drafts:
        row = np.full((1, width), -1, np.int32)
        row[0, :len(d)] = d
        out = oracle.pool_append(pool, plen, row)
        pool, plen = out["pool"], out["pool_len"]
        statuses.append(int(out["status"][0]))
    return pool, plen, statuses


def test_pool_append_case_study():
    pool, plen, st = _append_all(CASE_DRAFTS, len(CASE_POOL))
    assert plen[0] == len(CASE_POOL) and st == [0, 0, 0, 0]
    assert pool[0].tolist() == CASE_POOL
    # one slot short: the last draft does not fit and nothing of it is written
    pool, plen, st = _append_all(CASE_DRAFTS, len(CASE_POOL) - 1)
    assert st == [0, 0, 0, 128] and plen[0] == len(CASE_POOL) - 2
    assert pool[0, :plen[0]].tolist() == CASE_POOL[:-2] and pool[0, -1] == -7
    # an empty draft inserts nothing; a negative id ends a draft early
    pool, plen, st = _append_all([[], [5, 6, -1, 7]], 8)
    assert st == [0, 0] and plen[0] == 3 and pool[0, :3].tolist() == [5, 6, -1]


@pytest.mark.parametrize(
    "suffix, n, cont",
    [
        # "sure <call> find (": the whole suffix matches chunk 2's draft, whose rest is the call
        ([SURE, CALL, FIND, LP], 4, [TYO, COMMA, FRI, RP, ENDCALL]),
        # a shorter output: "<call> find (" matches both drafts; the later one (chunk 3) wins
        ([-1, CALL, FIND, LP], 3, [TYO]),
        # "find ( TYO": chunk 3's occurrence ends its draft, so only chunk 2 continues
        ([99, FIND, LP, TYO], 3, [COMMA, FRI, RP, ENDCALL]),
        # a mismatch at the oldest suffix token: only the two newest count
        ([99, 98, LP, TYO], 2, [COMMA, FRI, RP, ENDCALL]),
        # "</call>" and "ok" end their drafts: nothing follows them
        ([FRI, RP, ENDCALL, ENDCALL], 0, []),
        ([SURE, CALL, FIND, OK], 0, []),
        ([99, 99, 99, 99], 0, []),
        ([-1, -1, -1, -1], 0, []),
    ],
)
def test_pool_lookup_case_study(suffix, n, cont):
    gamma = 8
    out = oracle.pool_lookup(np.array([CASE_POOL], np.int32), np.array([len(CASE_POOL)], np.int32),
                             np.array([suffix], np.int32), gamma)
    assert out["match_len"][0] == n
    assert out["cont"][0].tolist() == cont + [-1] * (gamma - len(cont))
    # gamma caps the continuation; gamma 0 still reports the match
    out = oracle.pool_lookup(np.array([CASE_POOL], np.int32), np.array([len(CASE_POOL)], np.int32),
                             np.array([suffix], np.int32), 2)
    assert out["cont"][0].tolist() == (cont + [-1, -1])[:2]
    out = oracle.pool_lookup(np.array([CASE_POOL], np.int32), np.array([len(CASE_POOL)], np.int32),
                             np.array([suffix], np.int32), 0)
    assert out["match_len"][0] == n and out["cont"].shape == (1, 0)


def _ngram_index(drafts, N):
    """An n-gram index built the way the pages describe the pool: every n-gram
    (1 <= n <= N) of every draft that has a next token maps to (insertion rank,
    position of that next token); later insertions overwrite earlier ones."""
    index = {}
    rank = 0
    for d in drafts:
        for end in range(len(d) - 1):  # d[end + 1] exists
            for n in range(1, min(N, end + 1) + 1):
                index[tuple(d[end - n + 1:end + 1])] = (rank, d, end + 1)
            rank += 1
    return index


def test_pool_lookup_equals_an_ngram_index():
    rng = np.random.default_rng(11)
    for trial in range(300):
        vocab = int(rng.integers(2, 6))
        drafts = [rng.integers(0, vocab, int(rng.integers(0, 9))).tolist() for _ in range(int(rng.integers(0, 7)))]
        N = int(rng.integers(1, 6))
        gamma = int(rng.integers(0, 7))
        Lp = sum(len(d) + 1 for d in drafts if d) + int(rng.integers(0, 3))
        pool, plen, st = _append_all(drafts, max(Lp, 1), width=9)
        assert not any(st)
        out_len = int(rng.integers(0, N + 1))
        suffix = [-1] * (N - out_len) + rng.integers(0, vocab, out_len).tolist()
        got = oracle.pool_lookup(pool, plen, np.array([suffix], np.int32), gamma)
        index = _ngram_index([d for d in drafts if d], N)
        want_n, want = 0, []
        for n in range(out_len, 0, -1):
            hit = index.get(tuple(suffix[N - n:]))
            if hit is not None:
                _, d, start = hit
                want_n, want = n, d[start:start + gamma]
                break
        assert got["match_len"][0] == want_n, (trial, drafts, suffix)
        assert got["cont"][0].tolist() == want + [-1] * (gamma - len(want)), (trial, drafts, suffix)


def test_pool_lookup_continues_a_draft_the_output_follows():
    # Step 5: when the emitted output runs along a stored draft, the lookup hands
    # back the rest of that draft, so later forwards only pay for uncovered tokens.
    rng = np.random.default_rng(12)
    for _ in range(100):
        # distinct ids in every draft and no id shared between drafts: the match is unique
        drafts = [(2000 * j + rng.permutation(2000)[:int(rng.integers(2, 40))]).tolist() for j in range(5)]
        pool, plen, _ = _append_all(drafts, 256, width=40)
        j = int(rng.integers(0, 5))
        d = drafts[j]
        cut = int(rng.integers(1, len(d)))
        N = 6
        emitted = [10_001, 10_002] + d[:cut]  # tokens no draft holds, then the draft's prefix
        got = oracle.pool_lookup(pool, plen, np.array([emitted[-N:]], np.int32), 64)
        rest = d[cut:]
        assert got["match_len"][0] == min(cut, N)
        assert got["cont"][0].tolist() == rest + [-1] * (64 - len(rest))


def test_pool_lookup_pool_len_is_clamped():
    pool = np.array([[5, 6, 7, -1]], np.int32)
    for plen, n in [(-3, 0), (0, 0), (1, 0), (2, 1), (4, 1), (99, 1)]:
        got = oracle.pool_lookup(pool, np.array([plen], np.int32), np.array([[5]], np.int32), 4)
        assert got["match_len"][0] == n
        want = [6, 7][: max(0, min(plen, 4) - 1)] if n else []
        assert got["cont"][0].tolist() == want + [-1] * (4 - len(want))


def test_suffix_append_shifts_in_the_committed_tokens():
    # a step commits its n accepted drafts and the correction: tokens[0 .. n]
    suffix = np.array([[-1, -1, 5, 6], [1, 2, 3, 4], [9, 9, 9, 9]], np.int32)
    tokens = np.array([[7, 8, 9, -1], [10, -1, -1, -1], [20, 21, 22, 23]], np.int32)
    out = oracle.suffix_append(suffix, tokens, np.array([2, 0, 3], np.int32))
    assert out.tolist() == [[6, 7, 8, 9], [2, 3, 4, 10], [20, 21, 22, 23]]
    # accept lengths outside [0, k] are clamped; a longer commit than N keeps its last N tokens
    out = oracle.suffix_append(suffix[:1], np.array([[1, 2, 3, 4, 5, 6]], np.int32), np.array([99], np.int32))
    assert out.tolist() == [[3, 4, 5, 6]]
    out = oracle.suffix_append(suffix[:1], tokens[:1], np.array([-4], np.int32))
    assert out.tolist() == [[-1, 5, 6, 7]]


def test_verify_then_lookup_walks_along_a_stored_draft():
    # Steps 4 and 5 in a loop: each verify step commits a prefix of the pool's draft plus the
    # next token as its correction; the suffix update and the lookup then hand back the rest
    # of the draft after the committed tokens, until the draft is used up.
    rng = np.random.default_rng(14)
    for _ in range(50):
        drafts = [(3000 * j + rng.permutation(3000)[:int(rng.integers(10, 60))]).tolist() for j in range(4)]
        pool, plen, _ = _append_all(drafts, 512, width=60)
        d = drafts[int(rng.integers(0, 4))]
        N, k = 8, 6
        suffix = np.full((1, N), -1, np.int32)
        suffix[0, -1] = d[0]  # the output so far ends with the draft's first token
        pos = 1               # tokens of d emitted
        while True:
            got = oracle.pool_lookup(pool, plen, suffix, k)
            rest = d[pos:pos + k]
            assert got["cont"][0, :len(rest)].tolist() == rest
            if not rest:
                assert got["match_len"][0] == 0
                break
            n = int(rng.integers(0, len(rest)))  # drafts accepted; the next token is the correction
            tokens = np.full((1, k + 1), -1, np.int32)
            tokens[0, :n + 1] = d[pos:pos + n + 1]
            suffix = oracle.suffix_append(suffix, tokens, np.array([n], np.int32))
            pos += n + 1
            assert suffix[0, -1] == d[pos - 1]
