#!/usr/bin/env python3
"""Throughput of the speculative verify step on one GB300 (or N replicas).

One step = one call of the library on one batch of synthetic input already
resident in HBM.  The headline workload is the speculative-listening greedy
verify: 64 sessions x 65 target rows (a 32-token main draft plus a 32-token
runner-up branch) over V = 151,936 bf16 logits, 1.264 GB of logits per step,
more than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is logit GB/s (algorithmic bytes:
every logit row read once) summed over all ranks; `e2e` is the same metric
with the inputs copied from pinned host memory and the results read back
inside the timed region; `cpu_baseline` times the fp64 CPU oracle on a
bounded sample.  `--impl reference` times that oracle as the reference arm.

Launch: python bench.py [--steps K] [--warmup W]        (N = 1)
        python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["listen", "listen_top2", "d2t", "cfg", "sweep", "pool"], default="listen",
                    help="listen: greedy verify with a runner-up branch (headline); d2t: speculative sampling")
    ap.add_argument("--sessions", type=int, default=None,
                    help="requests per step (default: the workload's own, 64 listen sessions / 128 d2t requests)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true",
                    help="listen only: skip the d2t, CFG and sweep sub-records of the same line")
    ap.add_argument("--sub-steps", type=int, default=100, help="timed calls per sub-record")
    ap.add_argument("--cpu-seconds", type=float, default=16.0, help="CPU-baseline sample budget (two halves: "
                    "single-threaded, then all host threads)")
    return ap.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# GB300 HBM3e nominal bandwidth (the measured copy peak is the roofline denominator)
NOMINAL_HBM_GBS = 7900.0
# GB300 L2 capacity, and the buffer written to flush it
L2_BYTES = 129 << 20
L2_FLUSH_BYTES = 256 << 20


def _dist():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.sel = []
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid and not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            self.sel = ["-i", uuid] if uuid else []
        except Exception:
            self.sel = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.6)  # let the sampler start before the timed region
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            return None
        return rows

    @staticmethod
    def summarize(rows, t_first=None):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if re.match(r"^[0-9.]+$", r[1])]
        mx = [float(r[2]) for r in rows if re.match(r"^[0-9.]+$", r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
SAMPLING = ("d2t", "cfg")  # sampling workloads besides the sweep points


class Spec:
    """The inputs of one workload (seeded, synthetic, generated with torch on `device`),
    the algorithmic bytes one call must read, and its description.  Holds no library
    object, so the reference arm can use it without loading the CUDA library."""

    def __init__(self, name, device, sessions=None):
        import workloads

        self.name = name
        self.sweep = name.startswith("sweep_")
        if name in ("listen", "listen_top2"):
            w = workloads.listen(device=device, R=sessions or 64)
            R, k = w["R"], w["k"]
            self.rows = R * (2 * k + 1)
            self.logit_bytes = self.rows * w["V"] * 2
            self.inputs = {"target": w["target"], "draft": w["draft"]}
            self.dtype = "bf16"
            self.desc = (f"listen: {R} sessions x (32 main + 32 runner-up drafts) = 65 rows x 151936 bf16 per "
                         f"session ({self.logit_bytes / 1e9:.3f} GB of logits per step)")
            self.metric = "verify logit GB/s (speculative-listening greedy verify, V=151936 bf16)"
            if name == "listen_top2":
                self.desc = self.desc.replace("listen:", "listen with every row's argmax and runner-up:")
                self.metric = "verify + top-2 logit GB/s (speculative-listening greedy verify, V=151936 bf16)"
        elif name == "d2t" or self.sweep:
            if self.sweep:  # sweep_<bf16|f32>_b<B>
                _, dt, b = name.split("_")
                import torch

                w = workloads.sweep_batch(int(b[1:]), torch.bfloat16 if dt == "bf16" else torch.float32,
                                          device=device)
                self.dtype = dt
            else:
                w = workloads.d2t_workload(device=device, R=sessions or 128)
                self.dtype = "bf16"
            R, k, V, Vd = w["R"], w["k"], w["V"], w["Vd"]
            es = w["target"].element_size()
            self.sampled = int((w["temperature"] > 0).sum().item())
            self.rows = R * (k + 1)
            self.logit_bytes = R * (k + 1) * V * es + self.sampled * k * Vd * es + Vd * 4
            self.inputs = {"target": w["target"], "draft_logits": w["draft_logits"], "d2t": w["d2t"],
                           "draft": w["draft"], "seeds": w["seeds"], "temperature": w["temperature"]}
            if self.sweep:
                self.desc = (f"sweep point: {R} requests x (8 drafts + bonus) over V=151936 {dt}, half greedy, half "
                             f"sampled at T 0.6 / 1.0 with the d2t draft model (32000 ids) "
                             f"({self.logit_bytes / 1e9:.3f} GB of logits per call)")
                self.metric = f"verify+sample logit GB/s (sweep, {dt}, batch {R})"
            else:
                self.desc = (f"d2t: {R} requests x 7 drafts (+bonus) over V=151936 bf16, draft vocab 32000 bf16 "
                             f"via d2t, T=0.7 ({self.logit_bytes / 1e9:.3f} GB of logits per step; d2t plan built "
                             f"once per draft model, outside the step)")
                self.metric = "verify+sample logit GB/s (speculative sampling, d2t 32000 -> 151936, bf16)"
        elif name == "cfg":
            w = workloads.cfg_workload(device=device, R=sessions or 256)
            R, k, S, W = w["R"], w["k"], w["S"], w["W"]
            self.rows = R * (k + 1) * S
            self.logit_bytes = 2 * R * (k + 1) * S * W * 2 + R * k * S * W * 2
            self.inputs = {"cond": w["cond"], "uncond": w["uncond"], "draft_logits": w["draft_logits"],
                           "draft": w["draft"], "seeds": w["seeds"], "temperature": w["temperature"]}
            self.dtype = "bf16"
            self.desc = (f"cfg: {R} requests x {k} drafted frames (+1) x {S} codebooks of {W} bf16 entries, "
                         f"conditional + unconditional rows merged with w={w['w']}, T=1 "
                         f"({self.logit_bytes / 1e9:.3f} GB of logits per step)")
            self.metric = "CFG merge + verify logit GB/s (9 RVQ codebooks x 4096, bf16)"
        else:
            raise ValueError(name)
        self.w = w
        self._h = None

    # ---- the oracle side (host copies made once) ----
    def host(self):
        if self._h is None:
            import numpy as np

            import workloads

            w = self.w
            if self.name == "cfg":
                h = {"cond": workloads.host_rows(w["cond"]), "uncond": workloads.host_rows(w["uncond"]),
                     "draft_logits": workloads.host_rows(w["draft_logits"])}
            else:
                h = {"target": workloads.host_rows(w["target"])}
                if self.name not in ("listen", "listen_top2"):
                    h["draft_logits"] = workloads.host_rows(w["draft_logits"])
                    h["d2t"] = w["d2t"].cpu().numpy()
            h["draft"] = w["draft"].cpu().numpy()
            if "seeds" in w:
                h["seeds"] = w["seeds"].cpu().numpy().view(np.uint64)
                h["T"] = w["temperature"].cpu().numpy()
            self._h = h
        return self._h

    def oracle_one(self, r):
        """The oracle on request r: (its outputs, logit bytes, rows)."""
        import oracle

        w, h = self.w, self.host()
        k = w["k"]
        r = r % w["R"]
        if self.name in ("listen", "listen_top2"):
            rpr = 2 * k + 1
            out = oracle.verify_greedy(h["target"][r * rpr:(r + 1) * rpr], 1, k, 2, h["draft"][r:r + 1])
            if self.name == "listen_top2":
                oracle.top2_rows(h["target"][r * rpr:(r + 1) * rpr])
            return out, rpr * w["V"] * 2, rpr
        if self.name == "cfg":
            S, W = w["S"], w["W"]
            rr = (k + 1) * S
            out = oracle.cfg_merge_sample(h["cond"][r * rr:(r + 1) * rr], h["uncond"][r * rr:(r + 1) * rr],
                                          w["cb_id_base"], w["cb_data_offset"], S, W, w["w"],
                                          h["draft_logits"][r * k * S:(r + 1) * k * S], 1, k, h["draft"][r:r + 1],
                                          h["seeds"][r:r + 1], h["T"][r:r + 1])
            return out, 2 * rr * W * 2 + k * S * W * 2, rr
        es = h["target"].itemsize
        out = oracle.verify_sample(h["target"][r * (k + 1):(r + 1) * (k + 1)], h["draft_logits"][r * k:(r + 1) * k],
                                   h["d2t"], 1, k, h["draft"][r:r + 1], h["seeds"][r:r + 1], h["T"][r:r + 1])
        sampled = h["T"][r] > 0
        return out, (k + 1) * w["V"] * es + (k * w["Vd"] * es if sampled else 0), k + 1

    def oracle_requests(self, requests, threads):
        """The oracle over the given requests on `threads` host threads (the oracle is C called
        through ctypes, which releases the GIL): outputs concatenated in request order, bytes,
        rows, seconds."""
        import concurrent.futures as cf

        import numpy as np

        self.host()
        if not requests:
            return {}, 0, 0, 0.0
        t0 = time.perf_counter()
        if threads > 1:
            with cf.ThreadPoolExecutor(max_workers=threads) as ex:
                res = list(ex.map(self.oracle_one, requests))
        else:
            res = [self.oracle_one(r) for r in requests]
        el = time.perf_counter() - t0
        outs = {key: np.concatenate([o[key] for o, _, _ in res]) for key in res[0][0]}
        return outs, sum(b for _, b, _ in res), sum(n for _, _, n in res), el

    def oracle_sample(self, seconds, threads):
        """(GB/s, rows/s, requests, seconds) of the oracle over about `seconds` of requests,
        processed in rounds of `threads` requests at once."""
        self.host()
        done = nbytes = nrows = 0
        el = 0.0
        while el < seconds:
            _, b, n, t = self.oracle_requests(list(range(done, done + threads)), threads)
            done += threads
            nbytes += b
            nrows += n
            el += t
        return nbytes / el / 1e9, nrows / el, done, el


class Native:
    """The library call of one step on a Spec's device inputs: outputs, workspace, plan."""

    def __init__(self, spec, sv, device):
        import torch

        self.spec, self.sv = spec, sv
        w = spec.w
        R, k = w["R"], w["k"]
        i32 = dict(dtype=torch.int32, device=device)
        self.plan = None
        self.kernel_file, self.profile = None, None
        if spec.name in ("listen", "listen_top2"):
            self.out = dict(accept_len=torch.empty(R, **i32), tokens=torch.empty(R, k + 1, **i32),
                            branch=torch.empty(R, **i32), status=torch.empty(R, **i32))
            if spec.name == "listen":
                self.ws = torch.empty(sv.verify_greedy_workspace(R, k, 2, w["V"]), dtype=torch.uint8, device=device)
                self.launches = sv.LAUNCHES["verify_greedy"]
                self.kernel, self.profile = "argmax_segments_kernel<bf16>", "argmax_segments_listen.md"
            else:
                self.out["top2"] = torch.empty(spec.rows, 2, **i32)
                self.ws = torch.empty(sv.verify_greedy_top2_workspace(R, k, 2, w["V"]), dtype=torch.uint8,
                                      device=device)
                self.launches = sv.LAUNCHES["verify_greedy_top2"]
                self.kernel, self.profile = "argmax_segments_kernel<bf16, top-2>", "argmax_segments_listen_top2.md"
            self.kernel_file = "greedy.cu"
        elif spec.name == "cfg":
            S, W = w["S"], w["W"]
            self.out = dict(accept_len=torch.empty(R, **i32), tokens=torch.empty(R, k + 1, S, **i32),
                            status=torch.empty(R, **i32),
                            tv=torch.empty(R, k, S, dtype=torch.float32, device=device))
            self.ws = torch.empty(sv.cfg_merge_sample_workspace(R, k, S, W), dtype=torch.uint8, device=device)
            self.launches = sv.LAUNCHES["cfg_merge_sample"]
            self.kernel, self.kernel_file, self.profile = "cfg_rows_warp_kernel + cfg_race_kernel", "cfg.cu", \
                "cfg_rows_cfg.md"
        else:
            f32 = dict(dtype=torch.float32, device=device)
            self.out = dict(accept_len=torch.empty(R, **i32), tokens=torch.empty(R, k + 1, **i32),
                            status=torch.empty(R, **i32), tv=torch.empty(R, k, **f32),
                            p_draft=torch.empty(R, k, **f32), q_draft=torch.empty(R, k, **f32))
            self.ws = torch.empty(sv.verify_sample_workspace(R, k, w["V"], w["Vd"]), dtype=torch.uint8,
                                  device=device)
            # the d2t map is a constant of the draft model: its device plan is built once, here
            self.plan = sv.d2t_plan(w["d2t"], w["V"])
            self.launches = sv.LAUNCHES["verify_sample"]
            self.kernel, self.kernel_file = "sample_rows_fast_kernel + race_rows_kernel", "sample.cu"
            self.profile = "sample_rows_d2t.md" if spec.name == "d2t" else None

    def call(self, inp, stream):
        w, sv = self.spec.w, self.sv
        name = self.spec.name
        if name == "listen":
            sv.verify_greedy(inp["target"], w["R"], w["k"], 2, inp["draft"], out=self.out, workspace=self.ws,
                             stream=stream)
        elif name == "listen_top2":
            sv.verify_greedy_top2(inp["target"], w["R"], w["k"], 2, inp["draft"], out=self.out, workspace=self.ws,
                                  stream=stream)
        elif name == "cfg":
            sv.cfg_merge_sample(inp["cond"], inp["uncond"], w["cb_id_base"], w["cb_data_offset"], w["S"], w["W"],
                                w["w"], inp["draft_logits"], w["R"], w["k"], inp["draft"], inp["seeds"],
                                inp["temperature"], out=self.out, workspace=self.ws, stream=stream)
        else:
            sv.verify_sample(inp["target"], inp["draft_logits"], None, w["R"], w["k"], inp["draft"], inp["seeds"],
                             inp["temperature"], out=self.out, workspace=self.ws, stream=stream, plan=self.plan)


def _timed_calls(fn, steps, stream, flush):
    """Mean ms per call over `steps` calls on `stream`, each in its own CUDA events; with
    `flush`, an L2 flush (a write larger than L2) precedes every call outside its events;
    without, the calls run back to back inside one pair of events."""
    import torch

    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for f0_, f1_ in ev:
        flush.add_(1)
        f0_.record(stream)
        fn()
        f1_.record(stream)
    ev[-1][1].synchronize()
    return sum(f0_.elapsed_time(f1_) for f0_, f1_ in ev) / steps


def _sampling_stats(spec, out):
    """The pages' acceptance metrics of one call's outputs: per-position acceptance 1 - TV
    averaged over the sampled requests (raw_tv's complement; for CFG averaged over the
    codebooks too) and the mean accept length (drafts accepted per call)."""
    import numpy as np

    tv = out["tv"].float().cpu().numpy()
    n = out["accept_len"].cpu().numpy()
    T = spec.w["temperature"].cpu().numpy()
    s = T > 0
    tvs = tv[s].reshape(int(s.sum()), spec.w["k"], -1)
    return {"alpha_per_position": [round(float(a), 4) for a in 1.0 - tvs.mean(axis=(0, 2))],
            "mean_accept_len": float(n[s].mean()), "sampled_requests": int(s.sum())}


def _traffic_from_profile(kernel_file, profile):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel's file; None otherwise."""
    path = os.path.join(ROOT, "profiles", profile)
    src = os.path.join(ROOT, "serving_sampler_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        m = re.search(r"dram_bytes_per_launch:\s*([0-9]+)\s+source_sha256_16:\s*([0-9a-f]+)", text)
        if m and m.group(2) == digest:
            return int(m.group(1))
    except Exception:
        pass
    return None


def _oracle_threads():
    return max(1, os.cpu_count() or 1)


def run_reference(a):
    """Reference arm: the fp64 CPU oracle as it stands, on the host cores.  It loads the
    oracle only: the inputs come from the seeded generator (torch), never from the CUDA
    library."""
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch

    import oracle

    oracle.build()
    if a.workload == "pool":
        return _reference_pool(a, world)
    dev = "cuda" if torch.cuda.is_available() else "cpu"  # the generator's device: the native arm's bytes
    # the sweep's oracle leg times the sampling workload's requests (same step definition)
    spec = Spec("d2t" if a.workload == "sweep" else a.workload, dev, a.sessions)
    spec.host()
    threads = _oracle_threads()
    # one step = one round of `threads` requests, one per host thread
    spec.oracle_requests(list(range(threads * a.warmup)), threads)
    nbytes = nrows = 0
    el = 0.0
    for s_ in range(a.steps):
        lo = threads * (a.warmup + s_)
        _, b, n, t = spec.oracle_requests(list(range(lo, lo + threads)), threads)
        nbytes += b
        nrows += n
        el += t
    gbs = nbytes / el / 1e9
    done = a.steps * threads
    line = {
        "impl": "reference", "metric": spec.metric,
        "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": el / a.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.desc,
                   "step": f"{threads} requests of the workload through the CPU oracle, one per host thread",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{done} requests of the {a.workload} workload, {threads} per step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "rows_per_s": nrows / el,
    }
    print(json.dumps(line), flush=True)
    return 0


def _reference_pool(a, world):
    """Reference arm of the pool workload: the oracle's lookup over the 4096-session
    pools of the native arm's headline point, a bounded slice of 64 sessions per step."""
    import numpy as np

    import oracle
    import workloads

    R = 4096
    w = workloads.pool_session(R=R, seed=900 + R)
    pool = np.full((R, w["Lp"]), -1, np.int32)
    plen = np.zeros(R, np.int32)
    for d in w["drafts"][:-2]:
        o = oracle.pool_append(pool, plen, d)
        pool, plen = o["pool"], o["pool_len"]
    per = 64

    def one(s_):
        lo = (s_ * per) % R
        oracle.pool_lookup(pool[lo:lo + per], plen[lo:lo + per], w["suffix"][lo:lo + per], w["gamma"])

    for s_ in range(a.warmup):
        one(s_)
    t0 = time.perf_counter()
    for s_ in range(a.steps):
        one(a.warmup + s_)
    el = time.perf_counter() - t0
    v = a.steps * per / el
    line = {
        "impl": "reference", "metric": "hypothesis-pool lookups/s (longest 8-gram match, 32-token continuation)",
        "value": v, "unit": "lookups/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": el / a.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32", "data": "synthetic",
        "config": {"workload": "pool: the 4096-session pools, 64 sessions per step through the CPU oracle",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "lookups/s", "cores": 1, "kind": "oracle",
                         "sample": f"{a.steps * per} lookups, 64 per step"},
        "e2e": {"value": v, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


SUB_WORKLOADS = ("d2t", "cfg", "sweep_bf16_b1024", "sweep_bf16_b256")


def _roofline(spec, nat, ms, peak, peak_kind):
    achieved = spec.logit_bytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
            "traffic": _traffic_from_profile(nat.kernel_file, nat.profile) if nat.profile else None,
            "kernel": f"{nat.kernel} (all kernels of one call inside the same events)",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}


def _sub_record(name, sv, device, stream, steps, warmup, peak, peak_kind, flush, threads):
    """One sub-workload: timed calls (an L2 flush before every call), its roofline, the pages'
    acceptance metrics, and the oracle over every request for the exempt-row count."""
    import torch

    import oracle

    spec = Spec(name, device)
    nat = Native(spec, sv, device)
    fn = lambda: nat.call(spec.inputs, stream)  # noqa: E731
    for _ in range(max(warmup, 3)):
        fn()
    torch.cuda.synchronize()
    ms = _timed_calls(fn, steps, stream, flush)
    rec = {"metric": spec.metric, "value": spec.logit_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
           "us_per_call": ms * 1e3, "rows_per_s": spec.rows / (ms * 1e-3), "steps": steps,
           "workload": spec.desc, "l2": "flushed before every call, outside the timed events",
           "roofline": _roofline(spec, nat, ms, peak, peak_kind), "gpu_launches": steps * nat.launches}
    rec.update(_sampling_stats(spec, nat.out))
    # the oracle over the sampled requests: parity of tokens / accept lengths / status and the
    # rows whose decision margin is below 1e-6 (exempt from exact parity)
    T = spec.w["temperature"].cpu().numpy()
    req = [r for r in range(spec.w["R"]) if T[r] > 0]
    want, _, _, el = spec.oracle_requests(req, threads)
    got = {key: v.cpu().numpy()[req] for key, v in nat.out.items()}
    ex = oracle.exempt_rows(want)
    diff = (got["accept_len"] != want["accept_len"]) | np.any(
        got["tokens"].reshape(len(req), -1) != want["tokens"].reshape(len(req), -1), axis=1) | (
        got["status"] != want["status"])
    rec.update({"rows_checked": int(ex.size), "exempt_rows": int(ex.sum()),
                "requests_checked": len(req), "requests_differing": int(diff.sum()),
                "requests_differing_not_exempt": int((diff & ~ex.any(axis=1)).sum()),
                "oracle_seconds": round(el, 2), "oracle_threads": threads})
    del nat, spec
    torch.cuda.empty_cache()
    return rec


def run_native(a):
    import torch

    import serving_sampler_gb300 as sv
    from serving_sampler_gb300 import _build

    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: a CUDA GPU is required for the native arm")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    _barrier(world)
    sv.load()

    spec = Spec(a.workload, device, a.sessions)
    nat = Native(spec, sv, device)
    if torch.cuda.is_available():
        torch.cuda.empty_cache()  # drop the generator's fp32 temporaries
    stream = torch.cuda.current_stream(device)

    for _ in range(max(a.warmup, 3)):
        nat.call(spec.inputs, stream)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    # Inputs below four L2s get an L2 flush before every step, outside the events: the row
    # pass keeps the draft rows in L2 on purpose (for its TV pass), and back-to-back steps
    # would otherwise find them there.  Larger inputs run back to back.
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    _barrier(world)
    torch.cuda.synchronize()
    ms_local = _timed_calls(lambda: nat.call(spec.inputs, stream), a.steps, stream,
                            flush if spec.logit_bytes < 4 * L2_BYTES else None)
    _barrier(world)
    torch.cuda.synchronize()
    ms = _max_over_ranks(ms_local, world, device)
    value = world * spec.logit_bytes / (ms * 1e-3) / 1e9
    rows_per_s = world * spec.rows / (ms * 1e-3)
    peak, peak_kind = _peaks()
    roofline = _roofline(spec, nat, ms_local, peak, peak_kind)
    threads = _oracle_threads()

    # the sampling half of the metric: sub-records on the same box, in the same clock record
    subs = {}
    if rank == 0 and a.workload == "listen" and not a.no_sub:
        for name in SUB_WORKLOADS:
            subs[name] = _sub_record(name, sv, device, stream, max(3, min(a.steps, a.sub_steps)), a.warmup, peak,
                                     peak_kind, flush, threads)
    clock_rows = clocks.stop()
    del flush

    # end to end: pinned host inputs in, results out, every step
    e2e_steps = max(3, min(a.steps, 20))
    h_in = {}
    for key, t in spec.inputs.items():
        if t is None:
            continue
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        h_in[key] = h
    d_in = {key: torch.empty_like(spec.inputs[key]) for key in h_in}  # device buffers
    h_out = {key: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for key, v in nat.out.items()}

    def e2e_step():
        for key in d_in:
            d_in[key].copy_(h_in[key], non_blocking=True)
        nat.call(d_in, stream)
        for key, v in nat.out.items():
            h_out[key].copy_(v, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    _barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    f1.synchronize()
    _barrier(world)
    e2e_ms = _max_over_ranks(f0.elapsed_time(f1) / e2e_steps, world, device)
    h2d = sum(h.numel() * h.element_size() for h in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    e2e_value = world * spec.logit_bytes / (e2e_ms * 1e-3) / 1e9
    del h_in, d_in

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        g1, r1, d1, e1 = spec.oracle_sample(a.cpu_seconds / 2, 1)
        gn, rn, dn, en = spec.oracle_sample(a.cpu_seconds / 2, threads)
        cpu = {"value": gn, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{dn} requests of the {a.workload} workload in {en:.1f} s on {threads} host threads "
                         f"(one request per thread at a time), fp64 C as it stands",
               "rows_per_s": rn, "host_cores": os.cpu_count(),
               "single_thread": {"value": g1, "unit": "GB/s", "cores": 1, "rows_per_s": r1,
                                 "sample": f"{d1} requests in {e1:.1f} s"}}

    if rank == 0:
        line = {
            "metric": spec.metric,
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": spec.dtype, "data": "synthetic",
            "config": {"workload": spec.desc,
                       "l2": (f"inputs ({spec.logit_bytes / 1e9:.3f} GB) larger than 4 x L2 (129 MB); no flush"
                              if spec.logit_bytes >= 4 * L2_BYTES else
                              f"inputs ({spec.logit_bytes / 1e9:.3f} GB) below 4 x L2: L2 flushed before every "
                              f"step, outside the timed events"),
                       "parallelism": f"replicas x{world}"},
            "rows_per_s": rows_per_s,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps},
            "gpu_launches": a.steps * nat.launches,
            "clocks": Clocks.summarize(clock_rows),
        }
        if subs:
            line["sub"] = subs
            line["gpu_launches_sub"] = sum(r["gpu_launches"] for r in subs.values())
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_sweep(a):
    """Throughput sweep: batches {1, 8, 64, 256, 1024} x 9 positions (8 drafts + bonus),
    V = 151,936, bf16 and fp32 logits, half the requests greedy (T = 0) and half sampled
    (T alternating 0.6 / 1.0) with the d2t draft model of the sampling workload.  Every
    call is timed alone with CUDA events after an L2 flush.  Prints one JSON line with a
    point per (dtype, batch)."""
    import torch

    import serving_sampler_gb300 as sv
    import workloads
    from serving_sampler_gb300 import _build

    world, rank, local = _dist()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    _build.build()
    sv.load()
    stream = torch.cuda.current_stream(device)
    peak, peak_kind = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    k, V, Vd = 8, workloads.V_QWEN, workloads.VD_DRAFT
    steps = max(3, min(a.steps, 50))
    points = []
    clocks = Clocks(local)
    clocks.start()
    for dt, es in ((torch.bfloat16, 2), (torch.float32, 4)):
        for B in workloads.SWEEP_BATCHES:
            w = workloads.sweep_batch(B, dt, device=device)
            plan = sv.d2t_plan(w["d2t"], V)
            nsamp = int((w["temperature"] > 0).sum().item())
            nbytes = B * (k + 1) * V * es + nsamp * k * Vd * es
            out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=device),
                       tokens=torch.empty(B, k + 1, dtype=torch.int32, device=device),
                       status=torch.empty(B, dtype=torch.int32, device=device),
                       tv=torch.empty(B, k, dtype=torch.float32, device=device),
                       p_draft=torch.empty(B, k, dtype=torch.float32, device=device),
                       q_draft=torch.empty(B, k, dtype=torch.float32, device=device))
            ws = torch.empty(sv.verify_sample_workspace(B, k, V, Vd), dtype=torch.uint8, device=device)

            def call():
                sv.verify_sample(w["target"], w["draft_logits"], None, B, k, w["draft"], w["seeds"],
                                 w["temperature"], out=out, workspace=ws, stream=stream, plan=plan)

            for _ in range(max(a.warmup, 3)):
                call()
            torch.cuda.synchronize()
            # every call follows an L2 flush: the row pass keeps draft rows in L2 for its TV pass,
            # and without the flush a call could find the previous call's there
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in ev:
                flush.add_(1)
                e0.record(stream)
                call()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
            gbs = nbytes / (ms * 1e-3) / 1e9
            points.append({"dtype": "bf16" if es == 2 else "f32", "batch": B, "rows": B * (k + 1),
                           "sampled_requests": nsamp, "bytes": nbytes, "us_per_call": ms * 1e3, "GB/s": gbs,
                           "rows_per_s": B * (k + 1) / (ms * 1e-3), "roofline_frac": gbs / peak,
                           "l2": "flushed before each call"})
            del w, plan, out, ws
            torch.cuda.empty_cache()
    clock_rows = clocks.stop()
    best = max(p["GB/s"] for p in points)
    line = {
        "metric": "verify+sample logit GB/s sweep (batch x 9 positions, V=151936, 50/50 greedy/sampling)",
        "value": best, "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": max(a.warmup, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16,f32",
        "data": "synthetic",
        "config": {"workload": "sweep: batch {1,8,64,256,1024} x (8 drafts + bonus), d2t 32000 -> 151936, "
                               "T alternating 0 / 0.6 / 0 / 1.0 per request",
                   "value": "the best point"},
        "roofline_peak": {"value": peak, "unit": "GB/s",
                          "source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "fallback 6.8 TB/s"},
        "points": points,
        "gpu_launches": len(points) * (steps + max(a.warmup, 3)) * sv.LAUNCHES["verify_sample"],
        "clocks": Clocks.summarize(clock_rows),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_pool(a):
    """Hypothesis pool: sessions of 21 chunks, each inserting a main draft and a
    runner-up branch of up to 32 tokens (about 720 pool entries per session),
    then one lookup of the longest n-gram (N = 8) matching the emitted suffix
    with a 32-token continuation.  Per batch of sessions, the lookup call and the
    append call of one chunk are timed alone with CUDA events after an L2 flush.
    Prints one JSON line with a point per batch; bytes are the pool entries in
    use (int32) plus suffixes and continuations."""
    import torch

    import oracle
    import serving_sampler_gb300 as sv
    import workloads
    from serving_sampler_gb300 import _build

    world, rank, local = _dist()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    _build.build()
    sv.load()
    stream = torch.cuda.current_stream(device)
    peak, peak_kind = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    steps = max(3, min(a.steps, 50))
    points = []
    cpu = None
    clocks = Clocks(local)
    clocks.start()
    for R in (1, 64, 1024, 4096):
        w = workloads.pool_session(R=R, seed=900 + R)
        Lp, N, gamma = w["Lp"], w["N"], w["gamma"]
        pool = torch.full((R, Lp), -1, dtype=torch.int32, device=device)
        plen = torch.zeros(R, dtype=torch.int32, device=device)
        drafts = [torch.from_numpy(d).to(device) for d in w["drafts"]]
        for d in drafts[:-2]:
            sv.pool_append(pool, plen, d)
        suffix = torch.from_numpy(w["suffix"]).to(device)
        out = dict(match_len=torch.empty(R, dtype=torch.int32, device=device),
                   cont=torch.empty(R, gamma, dtype=torch.int32, device=device))
        used = int(plen.sum().item())
        look_bytes = 4 * (used + R + R * N + R + R * gamma)

        def timed(fn):
            for _ in range(max(a.warmup, 3)):
                fn()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in ev:
                flush.add_(1)
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize()
            return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps

        ms_look = timed(lambda: sv.pool_lookup(pool, plen, suffix, gamma, out=out, stream=stream))
        # append: the last chunk's main draft, undone after every call so the pool stays the same
        saved = plen.clone()

        def append():
            sv.pool_append(pool, plen, drafts[-2], stream=stream)
            plen.copy_(saved)

        ms_app = timed(append)
        gbs = look_bytes / (ms_look * 1e-3) / 1e9
        points.append({"sessions": R, "pool_entries": used, "lookup_us": ms_look * 1e3,
                       "lookups_per_s": R / (ms_look * 1e-3), "lookup_GB/s": gbs, "roofline_frac": gbs / peak,
                       "append_us_incl_restore_copy": ms_app * 1e3,
                       "matches": int((out["match_len"] > 0).sum().item())})
        if R == 64 and not a.no_cpu_baseline:
            pool_h, plen_h, suf_h = pool.cpu().numpy(), plen.cpu().numpy(), suffix.cpu().numpy()
            t0 = time.perf_counter()
            done = 0
            while time.perf_counter() - t0 < min(a.cpu_seconds, 5.0):
                oracle.pool_lookup(pool_h, plen_h, suf_h, gamma)
                done += R
            el = time.perf_counter() - t0
            cpu = {"value": done / el, "unit": "lookups/s", "cores": 1, "kind": "oracle",
                   "sample": f"{done} lookups of the 64-session pool, {el:.1f} s, single-threaded C"}
        del w, pool, plen, drafts, suffix, out
        torch.cuda.empty_cache()
    clock_rows = clocks.stop()
    big = points[-1]
    line = {
        "metric": "hypothesis-pool lookups/s (longest 8-gram match, 32-token continuation)",
        "value": big["lookups_per_s"], "unit": "lookups/s", "n_gpus": 1, "steps": steps,
        "warmup": max(a.warmup, 3), "ms_per_step": big["lookup_us"] * 1e-3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": "pool: sessions of 21 chunks x (main draft + runner-up), up to 32 tokens each, "
                               "N = 8, gamma = 32; value = the 4096-session point",
                   "l2": "flushed before each call"},
        "roofline_peak": {"value": peak, "unit": "GB/s",
                          "source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                          else "fallback 6.8 TB/s"},
        "points": points,
        "cpu_baseline": cpu,
        "gpu_launches": len(points) * 2 * (steps + max(a.warmup, 3)),
        "clocks": Clocks.summarize(clock_rows),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = _args()
    if a.impl == "reference":
        return run_reference(a)
    if a.workload == "sweep":
        return run_sweep(a)
    if a.workload == "pool":
        return run_pool(a)
    return run_native(a)


if __name__ == "__main__":
    sys.exit(main())
