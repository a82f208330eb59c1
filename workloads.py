"""Seeded synthetic inputs for the verify-and-sample workloads.

This module only draws inputs: logit rows, draft tokens, maps, seeds and
temperatures.  It holds none of the verification arithmetic (no softmax,
acceptance test, TV or sampler of the verifier).  Target argmax tokens are
planted, never searched; draft tokens come from a stand-in drafter that
draws from its own draft logits (Gumbel-max with torch's generator, or its
argmax for greedy requests).
Both the CUDA library's tests/benchmark and the CPU oracle read what it
produces, so the two sides always see the same bytes.

The stand-ins replace datasets and trained models that are not available
(TickTock-Bench sessions, DSpark / EAGLE3 draft models on a 151,936-token
target vocabulary, RVQ codec heads): shapes, vocabulary sizes, value
spread and acceptance profile follow the workload descriptions.

Workloads (names used by tests and the benchmark):
  tiny      4 requests x 8 drafts (+1 row), V = 4096, fp32 logits ~ N(0, 2^2);
            drafts = the planted argmax w.p. 0.7, else uniform; sampling
            variant with draft logits = target + N(0, 1), T = 1, seed 0.
  listen    64 sessions, a main draft of 32 tokens plus a 32-token runner-up
            branch (65 rows per session), V = 151,936 bf16 ~ N(0, 3^2) with
            the argmax planted 2.0 above the row maximum; 95% of main drafts
            match fully, 88% of the mismatches sit at position 0.
  d2t       128 requests x 7 drafts (+ bonus), V = 151,936 bf16, draft vocab
            32,000 with a seeded random injective d2t, T = 0.7.
  cfg       256 requests, 9 codebooks x 4096 entries, 4 drafted frames (+1),
            bf16 cond / uncond rows, w = 3, T = 1, flat distributions.
  pool      sessions of chunks whose drafts (a main draft of up to 32 tokens
            and a runner-up branch) are noisy windows of the session's final
            response, as in the tool-call case study: later chunks redraft
            what earlier ones already held; the emitted output is a prefix of
            the response, V = 151,936 token ids.
  sweep     batch x 9 rows (k = 8), V = 151,936, bf16 or fp32 ~ N(0, 3^2),
            requests alternating greedy (T = 0) and sampling (T in {0.6, 1.0})
            with d2t-truncated draft logits.
"""
from __future__ import annotations

import numpy as np
import torch

V_QWEN = 151_936
VD_DRAFT = 32_000


def splitmix64(x: int) -> int:
    """Seed scrambler for per-request Philox keys (Steele, Lea, Flood 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def seeds_array(base: int, R: int) -> np.ndarray:
    return np.array([splitmix64(base + r) for r in range(R)], dtype=np.uint64)


def seeds_tensor(base: int, R: int, device) -> torch.Tensor:
    """uint64 seeds stored in an int64 tensor (same bits)."""
    return torch.from_numpy(seeds_array(base, R).view(np.int64)).to(device)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _plant(z: torch.Tensor, idx: torch.Tensor, above: float) -> None:
    """Set z[i, idx[i]] = max_x z[i, x] + above (in place, fp32)."""
    rowmax = z.amax(dim=1)
    z.scatter_(1, idx.view(-1, 1), (rowmax + above).view(-1, 1))


def _rand_other(g, avoid: torch.Tensor, V: int) -> torch.Tensor:
    """Uniform token different from `avoid`, elementwise."""
    r = torch.randint(0, V - 1, avoid.shape, generator=g, device=avoid.device, dtype=torch.int64)
    return torch.where(r >= avoid, r + 1, r)


# ---------------------------------------------------------------------------
# greedy workloads
# ---------------------------------------------------------------------------
def greedy_batch(R: int, k: int, V: int, dtype=torch.bfloat16, sigma: float = 3.0, branches: int = 1,
                 p_full: float = 0.95, p_first: float = 0.88, seed: int = 0, device="cuda", row_pad: int = 0):
    """Target rows with planted argmaxes and drafts with a controlled accept profile.

    Returns dict(target [rows, V] (row stride V + row_pad), draft [R, branches, k], R, k, branches, V,
    planted [R, rows_per_request] argmax ids).
    """
    g = _gen(seed, device)
    rpr = 1 + branches * k
    rows = R * rpr
    z = torch.randn(rows, V + row_pad, generator=g, device=device, dtype=torch.float32) * sigma
    top = torch.randint(0, V, (rows,), generator=g, device=device)
    _plant(z[:, :V], top, 2.0)
    top = top.view(R, rpr)
    second = None
    if branches == 2:
        # second best of the shared first row: 1.0 above every other entry, 1.0 below the top
        second = _rand_other(g, top[:, 0], V)
        z0 = z.view(R, rpr, V + row_pad)[:, 0, :V]
        z0.scatter_(1, second.view(-1, 1), z0.gather(1, top[:, 0:1]) - 1.0)
    target = z.to(dtype)
    if row_pad:
        target = target[:, :V]
    # main branch: position j is verified by row j (row 0 shared with the runner-up)
    main = top[:, :k].clone()
    if k > 0:
        full = torch.rand(R, generator=g, device=device) < p_full
        first = torch.rand(R, generator=g, device=device) < p_first
        later = torch.randint(1, max(k, 2), (R,), generator=g, device=device).clamp(max=k - 1)
        pos = torch.where(first, torch.zeros_like(later), later)
        wrong = _rand_other(g, top.gather(1, pos.view(-1, 1)).view(-1), V)
        bad = ~full
        main[bad, pos[bad]] = wrong[bad]
    drafts = [main]
    if branches == 2:
        runner = torch.empty(R, k, dtype=torch.int64, device=device)
        # runner-up of row 0 excluding the main draft's first token
        runner[:, 0] = torch.where(main[:, 0] == top[:, 0], second, top[:, 0])
        runner[:, 1:] = top[:, k + 1:2 * k]
        drafts.append(runner)
    for b in range(1, branches) if branches > 2 else ():
        # tree drafts: branch b starts with the argmax of row 0 (viable) or another id, then
        # follows its own rows' argmaxes with one corrupted position w.p. 1/2
        br = top[:, b * k:b * k + k].clone()
        br[:, 0] = torch.where(torch.rand(R, generator=g, device=device) < 0.5, top[:, 0],
                               _rand_other(g, top[:, 0], V))
        if k > 1:
            pos = torch.randint(1, k, (R,), generator=g, device=device)
            bad = torch.rand(R, generator=g, device=device) < 0.5
            wrong = _rand_other(g, br.gather(1, pos.view(-1, 1)).view(-1), V)
            br[bad, pos[bad]] = wrong[bad]
        drafts.append(br)
    draft = torch.stack(drafts, dim=1).to(torch.int32).contiguous()
    return dict(target=target, draft=draft, R=R, k=k, branches=branches, V=V, planted=top)


def tiny_greedy(device="cuda", dtype=torch.float32):
    """4 requests x 8 drafts, V = 4096, fp32 ~ N(0, 2^2), drafts = argmax w.p. 0.7."""
    R, k, V = 4, 8, 4096
    g = _gen(0, device)
    rows = R * (k + 1)
    z = torch.randn(rows, V, generator=g, device=device) * 2.0
    top = torch.randint(0, V, (rows,), generator=g, device=device)
    _plant(z, top, 0.5)
    top = top.view(R, k + 1)
    keep = torch.rand(R, k, generator=g, device=device) < 0.7
    other = torch.randint(0, V, (R, k), generator=g, device=device)
    draft = torch.where(keep, top[:, :k], other).to(torch.int32).view(R, 1, k).contiguous()
    return dict(target=z.to(dtype), draft=draft, R=R, k=k, branches=1, V=V, planted=top)


def listen(device="cuda", R: int = 64, seed: int = 1236):
    """Speculative-listening greedy verify: 64 sessions x (32 main + 32 runner) drafts, 65 rows each."""
    return greedy_batch(R, 32, V_QWEN, torch.bfloat16, 3.0, branches=2, seed=seed, device=device)


def host_rows(t: torch.Tensor) -> np.ndarray:
    """A CPU numpy copy of logit rows: bf16 -> uint16 bit patterns, fp32 as is."""
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().contiguous().numpy()


# ---------------------------------------------------------------------------
# sampling workloads
# ---------------------------------------------------------------------------
# Support bias and per-position draft noise of the d2t workload, chosen by
# oracle/calibrate_d2t.py so that the mean off-support p-mass is about 0.10
# and the mean single-position acceptance 1 - TV follows the DSpark profile
# 0.714 ... 0.423 quoted in "speculative decoding for Omni models", section 3.
D2T_DELTA = 2.73
D2T_SIGMA = [0.48, 0.71, 0.9, 1.01, 1.12, 1.2, 1.27]


def _draw_drafts(g, y: torch.Tensor, T: torch.Tensor, greedy: torch.Tensor) -> torch.Tensor:
    """Draft ids from draft logits y [n, Vd]: Gumbel-max at temperature T (per row),
    or the argmax for greedy rows."""
    u = torch.rand(y.shape, generator=g, device=y.device).clamp_min_(1e-30)
    gumbel = -torch.log(-torch.log(u))
    Tpos = torch.where(T > 0, T, torch.ones_like(T)).view(-1, 1)
    noisy = y / Tpos + gumbel
    pick = torch.where(greedy.view(-1, 1), y, noisy)
    return pick.argmax(dim=1)


def sample_batch(R: int, k: int, V: int, Vd: int | None = None, dtype=torch.bfloat16, draft_dtype=None,
                 T=1.0, sigma_pos=1.0, delta: float = 0.0, z_sigma: float = 3.0, seed: int = 0,
                 seed_base: int = 1234, device="cuda", row_pad: int = 0, d2t_seed: int | None = None):
    """Target rows [R*(k+1), V], draft rows [R*k, Vd] (= target restricted to the d2t
    image, plus the support bias, plus N(0, sigma_j^2) noise), d2t (None when Vd is
    None: identity), drafts x_j drawn from the draft distribution at T, seeds, T."""
    draft_dtype = draft_dtype or dtype
    g = _gen(seed, device)
    rows = R * (k + 1)
    z = torch.randn(rows, V + row_pad, generator=g, device=device, dtype=torch.float32) * z_sigma
    d2t = None
    if Vd is not None:
        gd = _gen(seed + 7 if d2t_seed is None else d2t_seed, device)
        d2t = torch.randperm(V, generator=gd, device=device)[:Vd].to(torch.int32)
        z[:, d2t.long()] += delta
    else:
        Vd = V
    Tt = torch.as_tensor(T, dtype=torch.float32, device=device).expand(R).contiguous()
    sig = torch.as_tensor(sigma_pos, dtype=torch.float32, device=device).expand(k).contiguous()
    zr = z.view(R, k + 1, V + row_pad)[:, :k, :V]
    base = zr if d2t is None else zr[:, :, d2t.long()]
    noise = torch.randn(base.shape, generator=g, device=device) * sig.view(1, k, 1)
    y = (base + noise).reshape(R * k, Vd)
    target = z.to(dtype)
    if row_pad:
        target = target[:, :V]
    draft_logits = y.to(draft_dtype).contiguous()
    greedy = (Tt <= 0).repeat_interleave(k)
    ids = _draw_drafts(g, draft_logits.float(), Tt.repeat_interleave(k), greedy)
    draft = (ids if d2t is None else d2t.long()[ids]).view(R, k).to(torch.int32).contiguous()
    return dict(target=target, draft_logits=draft_logits, d2t=d2t, draft=draft,
                seeds=seeds_tensor(seed_base, R, device), temperature=Tt, R=R, k=k, V=V, Vd=Vd)


def tiny_sample(device="cuda"):
    """4 requests x 8 drafts, V = 4096 fp32 ~ N(0, 2^2), draft logits = target + N(0, 1), T = 1, seed 0."""
    return sample_batch(4, 8, 4096, None, torch.float32, T=1.0, sigma_pos=1.0, z_sigma=2.0, seed=0,
                        seed_base=0, device=device)


def d2t_workload(device="cuda", R: int = 128, batch: int = 0):
    """128 requests x 7 drafts (+ bonus), V = 151,936 bf16, draft vocabulary 32,000 via a seeded
    random injective d2t, T = 0.7, per-request seeds splitmix64(1234 + r).  `batch` > 0 draws
    another batch of the same configuration (other logits, drafts and request seeds; the same
    d2t map, a constant of the draft model)."""
    return sample_batch(R, 7, V_QWEN, VD_DRAFT, torch.bfloat16, T=0.7, sigma_pos=D2T_SIGMA,
                        delta=D2T_DELTA, z_sigma=3.0, seed=1237 + 7919 * batch,
                        seed_base=1234 + 1_000_003 * batch, device=device, d2t_seed=1244)


SWEEP_BATCHES = (1, 8, 64, 256, 1024)


def sweep_batch(B: int, dtype=torch.bfloat16, device="cuda"):
    """A point of the throughput sweep: B requests x (8 drafts + bonus), V = 151,936, the d2t
    draft model of the sampling workload, requests alternating greedy (T = 0) and sampled
    (T alternating 0.6 / 1.0)."""
    T = [0.0 if r % 2 == 0 else (0.6 if (r // 2) % 2 == 0 else 1.0) for r in range(B)]
    sigma = list(D2T_SIGMA) + [D2T_SIGMA[-1]]
    return sample_batch(B, 8, V_QWEN, VD_DRAFT, dtype, T=T, sigma_pos=sigma, delta=D2T_DELTA, z_sigma=3.0,
                        seed=1300 + B, seed_base=5000, device=device)


# ---------------------------------------------------------------------------
# CFG workload
# ---------------------------------------------------------------------------
CFG_TEXT_V = V_QWEN - 9 * 4096  # text partition size; audio codebook s starts at CFG_TEXT_V + 4096 s


def cfg_batch(R: int, k: int, S: int, W: int, w: float = 3.0, T=1.0, dtype=torch.bfloat16, draft_dtype=None,
              sigma_h: float = 0.5, sigma_e: float = 0.1, bump: float = 7.1, sigma_d: float = 1.0,
              seed: int = 0, seed_base: int = 1234, device="cuda", row_len: int | None = None,
              offsets=None, greedy_drafts: float = 0.0):
    """cond / uncond rows [R*(k+1)*S, row_len] (codebook s at offsets[s], W entries):
    c = h + e_c, u = h + e_u with a shared component h ~ N(0, sigma_h^2) and e ~ N(0, sigma_e^2);
    one id per row is planted `bump` above h so the guided distribution has a top-1 near 0.2
    (flat RVQ codebooks).  Draft rows [R*k*S, W] = the guided latent + N(0, sigma_d^2); drafts
    are drawn from them (absolute ids cb_id_base[s] + local)."""
    draft_dtype = draft_dtype or dtype
    g = _gen(seed, device)
    rows = R * (k + 1) * S
    row_len = row_len or W
    offsets = list(offsets) if offsets is not None else [0] * S
    h = torch.randn(rows, W, generator=g, device=device) * sigma_h
    top = torch.randint(0, W, (rows,), generator=g, device=device)
    h.scatter_add_(1, top.view(-1, 1), torch.full((rows, 1), bump, device=device))
    ec = torch.randn(rows, W, generator=g, device=device) * sigma_e
    eu = torch.randn(rows, W, generator=g, device=device) * sigma_e
    cond = torch.randn(rows, row_len, generator=g, device=device)
    uncond = torch.randn(rows, row_len, generator=g, device=device)
    svec = torch.arange(rows, device=device) % S
    for s in range(S):
        sel = svec == s
        cond[sel, offsets[s]:offsets[s] + W] = h[sel] + ec[sel]
        uncond[sel, offsets[s]:offsets[s] + W] = h[sel] + eu[sel]
    guided = (h + w * ec - (w - 1.0) * eu).view(R, k + 1, S, W)[:, :k]
    y = (guided + torch.randn(guided.shape, generator=g, device=device) * sigma_d).reshape(R * k * S, W)
    draft_logits = y.to(draft_dtype).contiguous()
    Tt = torch.as_tensor(T, dtype=torch.float32, device=device).expand(R).contiguous()
    greedy = torch.rand(R * k * S, generator=g, device=device) < greedy_drafts
    ids = _draw_drafts(g, draft_logits.float(), Tt.repeat_interleave(k * S), greedy)
    base = torch.tensor([CFG_TEXT_V + 4096 * s for s in range(S)], dtype=torch.int64, device=device)
    draft = (ids.view(R, k, S) + base.view(1, 1, S)).to(torch.int32).contiguous()
    return dict(cond=cond.to(dtype), uncond=uncond.to(dtype), draft_logits=draft_logits, draft=draft,
                cb_id_base=base.tolist(), cb_data_offset=offsets, S=S, W=W, w=w, R=R, k=k,
                seeds=seeds_tensor(seed_base, R, device), temperature=Tt)


def cfg_workload(device="cuda", R: int = 256, batch: int = 0):
    """256 requests, 9 codebooks x 4096 entries, 4 drafted frames (+1), bf16, w = 3, T = 1;
    `batch` > 0 draws another batch of the same configuration."""
    return cfg_batch(R, 4, 9, 4096, 3.0, 1.0, torch.bfloat16, seed=1238 + 7919 * batch,
                     seed_base=1234 + 3 + 1_000_003 * batch, device=device)


def pool_session(R: int = 64, chunks: int = 21, gamma: int = 32, N: int = 8, V: int = 151936, seed: int = 77,
                 noise: float = 0.05):
    """Hypothesis-pool inputs: per chunk a main draft and a runner-up branch per
    session (int32 [R, gamma], -1 padded), and the emitted suffix int32 [R, N].

    Session r has a final response of 4 * gamma tokens.  Chunk c's main draft is
    a window of it that starts near the response's beginning and grows with c,
    cut to a random length, with each token replaced by a random id w.p.
    `noise`; the runner-up branch is random ids of random length.  The emitted
    output is a random prefix of the response (at least one token)."""
    rng = np.random.default_rng(seed)
    L = 4 * gamma
    resp = rng.integers(0, V, (R, L), dtype=np.int64)
    drafts = []
    for c in range(chunks):
        for branch in range(2):
            d = np.full((R, gamma), -1, np.int64)
            for r in range(R):
                n = int(rng.integers(1, gamma + 1))
                if branch == 0:
                    start = int(rng.integers(0, min(L - n, 2 * c + 1) + 1))
                    tok = resp[r, start:start + n].copy()
                    flip = rng.random(n) < noise
                    tok[flip] = rng.integers(0, V, int(flip.sum()))
                else:
                    tok = rng.integers(0, V, n)
                d[r, :n] = tok
            drafts.append(d.astype(np.int32))
    emitted = rng.integers(1, L, R)
    suffix = np.full((R, N), -1, np.int32)
    for r in range(R):
        tail = resp[r, max(0, emitted[r] - N):emitted[r]]
        suffix[r, N - len(tail):] = tail
    Lp = chunks * 2 * (gamma + 1)
    return dict(drafts=drafts, suffix=suffix, Lp=Lp, R=R, N=N, gamma=gamma)
