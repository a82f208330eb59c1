"""Every entry point on seeded random configurations against the oracle.  Speculative and CFG
sampling: both dtypes and their mixes, widths that are and are not multiples of the 16-byte
vector, the identity map and d2t maps of every density, codebook counts and widths, k from 0 to
9, batches of 1 to 12 requests with greedy, sampled and invalid temperatures mixed (the bulk-copy
row pass and the general one, race partitions that cut rows at odd places).  Greedy verification
with branches and tree drafts, NaN / +-inf rows and planted ties, with and without the top-2
output; modality inference over random partitions; the accept scan; hypothesis-pool sessions.
Sampling outputs follow the parity rules (tokens, accept lengths and status exact outside the
decision margin; TV, p and q within 1e-5 relative), everything else is compared exactly."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.sampling_parity import compare
from tests.test_gpu_cfg import _oracle as _cfg_oracle
from tests.test_gpu_cfg import _run as _cfg_run
from tests.test_gpu_sample import _oracle, _run

pytestmark = pytest.mark.gpu

DTYPES = (torch.bfloat16, torch.float32)
TEMPS = (0.0, 0.3, 0.7, 1.0, 1.6, -0.5)  # a negative temperature: verified greedily, flagged


def case(i: int):
    """The i-th configuration (a pure function of i)."""
    rng = np.random.default_rng(9100 + i)
    dt = DTYPES[rng.integers(2)]
    dd = DTYPES[rng.integers(2)] if rng.random() < 0.3 else dt
    V = int(rng.choice([int(rng.integers(9, 600)), int(rng.integers(600, 20000))]))
    Vd = None if rng.random() < 0.3 else int(rng.integers(1, min(V, 4000) + 1))
    if rng.random() < 0.5:  # widths in whole 16-byte vectors (the bulk-copy path when the map is given)
        V = max(8, V // 8 * 8)
        Vd = None if Vd is None else max(8, min(V, Vd) // 8 * 8)
    k = int(rng.integers(0, 10))
    R = int(rng.integers(1, 13))
    T = [float(TEMPS[j]) for j in rng.integers(0, len(TEMPS), R)]
    return dict(R=R, k=k, V=V, Vd=Vd, dtype=dt, draft_dtype=dd, T=T,
                sigma_pos=float(rng.uniform(0.2, 1.5)), delta=float(rng.uniform(0, 3)) if Vd else 0.0,
                z_sigma=float(rng.uniform(0.5, 4)), seed=int(rng.integers(1 << 30)),
                seed_base=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("i", range(32))
def test_random_configuration(sv, i):
    c = case(i)
    w = workloads.sample_batch(c["R"], c["k"], c["V"], c["Vd"], c["dtype"], c["draft_dtype"], T=c["T"],
                               sigma_pos=c["sigma_pos"], delta=c["delta"], z_sigma=c["z_sigma"], seed=c["seed"],
                               seed_base=c["seed_base"])
    compare(_run(sv, w), _oracle(w), label=f"fuzz {i}")


def test_cases_cover_both_row_passes():
    """The configurations reach the bulk-copy row pass (matched dtypes, a d2t map, widths that are
    multiples of eight) and the general one (identity, mixed dtypes, odd widths)."""
    fast = general = 0
    for i in range(32):
        c = case(i)
        ok = c["Vd"] is not None and c["dtype"] == c["draft_dtype"] and c["V"] % 8 == 0 and c["Vd"] % 8 == 0
        fast += ok
        general += not ok
    assert fast >= 4 and general >= 4, (fast, general)


def cfg_case(i: int):
    """The i-th CFG configuration (a pure function of i)."""
    rng = np.random.default_rng(9300 + i)
    dt = DTYPES[rng.integers(2)]
    dd = DTYPES[rng.integers(2)] if rng.random() < 0.3 else dt
    R, k, S = int(rng.integers(1, 11)), int(rng.integers(0, 7)), int(rng.integers(1, 17))
    W = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 6000))]))
    T = [float(TEMPS[j]) for j in rng.integers(0, len(TEMPS), R)]
    return dict(R=R, k=k, S=S, W=W, w=float(rng.uniform(1.0, 5.0)), T=T, dtype=dt, draft_dtype=dd,
                sigma_h=float(rng.uniform(0.2, 1.0)), bump=float(rng.uniform(0.0, 8.0)),
                sigma_d=float(rng.uniform(0.3, 1.5)), greedy_drafts=float(rng.uniform(0, 0.5)),
                seed=int(rng.integers(1 << 30)), seed_base=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("i", range(16))
def test_random_cfg_configuration(sv, i):
    c = cfg_case(i)
    w = workloads.cfg_batch(c["R"], c["k"], c["S"], c["W"], c["w"], c["T"], c["dtype"], c["draft_dtype"],
                            sigma_h=c["sigma_h"], bump=c["bump"], sigma_d=c["sigma_d"], seed=c["seed"],
                            seed_base=c["seed_base"], greedy_drafts=c["greedy_drafts"])
    compare(_cfg_run(sv, w), _cfg_oracle(w), label=f"cfg fuzz {i}")


def greedy_case(i: int):
    """The i-th greedy configuration (a pure function of i)."""
    rng = np.random.default_rng(9500 + i)
    branches = int(rng.choice([1, 1, 2, 3, 8]))
    k = int(rng.integers(1 if branches > 1 else 0, 41))
    V = int(rng.choice([int(rng.integers(2, 700)), int(rng.integers(700, 30000)), workloads.V_QWEN]))
    return dict(R=int(rng.integers(1, 41)), k=k, branches=branches, V=V, dtype=DTYPES[rng.integers(2)],
                row_pad=int(rng.choice([0, 0, int(rng.integers(1, 9))])), p_full=float(rng.uniform(0.2, 1.0)),
                p_first=float(rng.uniform(0.2, 1.0)), seed=int(rng.integers(1 << 30)),
                specials=int(rng.integers(0, 4)), ties=bool(rng.random() < 0.5), rng_seed=9700 + i)


@pytest.mark.parametrize("i", range(24))
def test_random_greedy_configuration(sv, i):
    """Greedy verification (branches and tree drafts), and the same call with every row's argmax and
    runner-up, on random shapes with NaN / +-inf rows and planted ties."""
    from tests.test_gpu_greedy import _check, _check_top2

    c = greedy_case(i)
    w = workloads.greedy_batch(c["R"], c["k"], c["V"], c["dtype"], branches=c["branches"], p_full=c["p_full"],
                               p_first=c["p_first"], seed=c["seed"], row_pad=c["row_pad"])
    t = w["target"].float()
    rng = np.random.default_rng(c["rng_seed"])
    rows = t.shape[0]
    for _ in range(c["specials"]):  # a NaN, +inf or -inf at a random place, or a row of -inf
        r, x = int(rng.integers(rows)), int(rng.integers(c["V"]))
        kind = int(rng.integers(4))
        if kind == 3:
            t[r, :] = float("-inf")
        else:
            t[r, x] = (float("nan"), float("inf"), float("-inf"))[kind]
    if c["ties"]:  # a copy of a row's maximum at a random other id
        for r in rng.integers(0, rows, size=min(rows, 5)):
            m = int(torch.argmax(torch.nan_to_num(t[r], nan=-float("inf"))).item())
            t[int(r), int(rng.integers(c["V"]))] = t[int(r), m]
    target = t.to(c["dtype"])
    if c["row_pad"]:  # keep the padded row stride of the generator
        full = torch.empty(rows, c["V"] + c["row_pad"], dtype=c["dtype"], device=target.device)
        full[:, :c["V"]] = target
        target = full[:, :c["V"]]
    _check(sv, target, c["R"], c["k"], c["branches"], w["draft"])
    _check_top2(sv, target, c["R"], c["k"], c["branches"], w["draft"])


@pytest.mark.parametrize("i", range(12))
def test_random_modality_and_accept_scan(sv, i):
    rng = np.random.default_rng(9900 + i)
    dtype = DTYPES[rng.integers(2)]
    N, V = int(rng.integers(1, 200)), int(rng.integers(2, 40000))
    P = int(rng.integers(1, 65))
    starts = np.sort(rng.integers(0, V + 1, P)).astype(np.int32)
    g = torch.Generator(device="cuda").manual_seed(int(rng.integers(1 << 30)))
    z = (torch.randn(N, V, generator=g, device="cuda") * float(rng.uniform(0.5, 5))).to(dtype)
    got = sv.infer_modality(z, starts.tolist())
    torch.cuda.synchronize()
    want = oracle.infer_modality(workloads.host_rows(z), starts)
    for key in ("amax", "part", "mask_lo", "mask_hi"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), want[key], err_msg=key)
    R, k = int(rng.integers(1, 60)), int(rng.integers(1, 257))
    acc = (rng.random((R, k)) < float(rng.uniform(0.3, 1.0))).astype(np.uint8)
    draft = rng.integers(0, 5000, (R, k)).astype(np.int32)
    fix = rng.integers(0, 5000, (R, k + 1)).astype(np.int32)
    got = sv.accept_scan(torch.from_numpy(acc).cuda(), torch.from_numpy(draft).cuda(), torch.from_numpy(fix).cuda())
    torch.cuda.synchronize()
    want = oracle.accept_scan(acc, draft, fix)
    np.testing.assert_array_equal(got["accept_len"].cpu().numpy(), want["accept_len"])
    np.testing.assert_array_equal(got["tokens"].cpu().numpy(), want["tokens"])


@pytest.mark.parametrize("i", range(12))
def test_random_pool_sessions(sv, i):
    """Hypothesis pools: appends of random draft blocks (negative ids end a draft early), lookups
    of the emitted suffix, suffix updates with accept lengths inside and outside [0, k]."""
    from tests.test_gpu_pool import _append_both, _dev, _lookup_both

    rng = np.random.default_rng(10100 + i)
    R, Lp, vocab = int(rng.integers(1, 300)), int(rng.integers(0, 5000)), int(rng.integers(2, 60))
    N, gamma = int(rng.integers(0, 65)), int(rng.integers(0, 257))
    pool_h = np.full((R, Lp), -2, np.int32)
    plen_h = np.zeros(R, np.int32)
    pool_d, plen_d = _dev(pool_h), _dev(plen_h)
    suffix = rng.integers(-1, vocab, (R, N)).astype(np.int32)
    for step in range(int(rng.integers(1, 8))):
        k = int(rng.integers(0, 41))
        drafts = rng.integers(0, vocab, (R, k)).astype(np.int32)
        if k:
            cut = rng.random(R) < 0.3  # some drafts end early
            drafts[cut, int(rng.integers(k))] = -1
        pool_h, plen_h = _append_both(sv, pool_d, plen_d, pool_h, plen_h, drafts)
        _lookup_both(sv, pool_h, plen_h, suffix, gamma, pool_d, plen_d)
        tokens = rng.integers(0, vocab, (R, k + 1)).astype(np.int32)
        acc = rng.integers(-2, k + 3, R).astype(np.int32)
        s_d = _dev(suffix)
        sv.suffix_append(s_d, _dev(tokens), _dev(acc))
        want = oracle.suffix_append(suffix, tokens, acc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(s_d.cpu().numpy(), want, err_msg=f"suffix after step {step}")
        suffix = want


@pytest.mark.parametrize("i", range(8))
def test_random_long_draft_blocks(sv, i):
    """Sampling and CFG with k from 10 to 256 (scans over several 32-position words)."""
    rng = np.random.default_rng(10300 + i)
    dt = DTYPES[rng.integers(2)]
    k = int(rng.integers(10, 257))
    R = int(rng.integers(1, 5))
    V = int(rng.choice([int(rng.integers(8, 300)), 8 * int(rng.integers(8, 400))]))
    Vd = None if rng.random() < 0.4 else max(1, int(rng.integers(1, V + 1)) // 8 * 8)
    T = [float(TEMPS[j]) for j in rng.integers(0, len(TEMPS), R)]
    # drafts close to the target: long accepted runs
    w = workloads.sample_batch(R, k, V, Vd, dt, T=T, sigma_pos=float(rng.uniform(0.01, 0.3)), delta=1.0 if Vd else 0.0,
                               z_sigma=float(rng.uniform(0.5, 3)), seed=int(rng.integers(1 << 30)),
                               seed_base=int(rng.integers(1 << 30)))
    compare(_run(sv, w), _oracle(w), label=f"long k {i}")
    S, W = int(rng.integers(1, 5)), int(rng.integers(2, 600))
    kc = int(rng.integers(10, 65))
    wc = workloads.cfg_batch(R, kc, S, W, float(rng.uniform(1, 4)), T, dt, sigma_h=0.5, bump=float(rng.uniform(4, 12)),
                             sigma_d=0.05, seed=int(rng.integers(1 << 30)), seed_base=int(rng.integers(1 << 30)))
    compare(_cfg_run(sv, wc), _cfg_oracle(wc), label=f"long k cfg {i}")
