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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["listen"], default="listen")
    ap.add_argument("--sessions", type=int, default=64, help="listen sessions per step (64 = the workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    return ap.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


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
def _listen(device, sessions=64):
    import torch

    import workloads

    w = workloads.listen(device=device, R=sessions)
    if torch.cuda.is_available():
        torch.cuda.empty_cache()  # drop the generator's fp32 temporaries
    R, k = w["R"], w["k"]
    rows = R * (2 * k + 1)
    V = w["V"]
    logit_bytes = rows * V * 2  # bf16, every row read once
    return w, dict(R=R, k=k, rows=rows, V=V, logit_bytes=logit_bytes)


def _traffic_from_profile(kernel_file):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel's file; None otherwise."""
    path = os.path.join(ROOT, "profiles", "argmax_segments_listen.md")
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


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample
# ---------------------------------------------------------------------------
def _oracle_sample(host_target, draft_np, meta, seconds, max_requests=None):
    """Run the oracle request by request until `seconds` of CPU work; returns
    (GB/s, rows/s, requests done, seconds)."""
    import oracle

    R, k = meta["R"], meta["k"]
    rpr = 2 * k + 1
    done = 0
    t0 = time.perf_counter()
    while True:
        r = done % R
        oracle.verify_greedy(host_target[r * rpr:(r + 1) * rpr], 1, k, 2, draft_np[r:r + 1])
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_requests is not None and done >= max_requests):
            break
    bytes_done = done * rpr * meta["V"] * 2
    return bytes_done / el / 1e9, done * rpr / el, done, el


def run_reference(a):
    """Reference arm: the fp64 CPU oracle as it stands, one request per step."""
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    import torch

    import workloads

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w, meta = _listen(dev, a.sessions)
    host = workloads.host_rows(w["target"])
    draft = w["draft"].cpu().numpy()
    del w
    import oracle

    oracle.build()
    k, rpr = meta["k"], 2 * meta["k"] + 1
    for s in range(a.warmup):
        r = s % meta["R"]
        oracle.verify_greedy(host[r * rpr:(r + 1) * rpr], 1, k, 2, draft[r:r + 1])
    t0 = time.perf_counter()
    for s in range(a.steps):
        r = s % meta["R"]
        oracle.verify_greedy(host[r * rpr:(r + 1) * rpr], 1, k, 2, draft[r:r + 1])
    el = time.perf_counter() - t0
    step_bytes = rpr * meta["V"] * 2
    gbs = a.steps * step_bytes / el / 1e9
    line = {
        "impl": "reference", "metric": "verify logit GB/s (speculative-listening greedy verify, V=151936 bf16)",
        "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": el / a.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "listen: 64 sessions x (32 main + 32 runner-up drafts), 65 rows x 151936 bf16",
                   "step": "one session (65 rows) through the CPU oracle", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{a.steps} sessions of the listen workload, one per step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "rows_per_s": a.steps * rpr / el,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_native(a):
    import torch

    import serving_sampler_gb300 as sv
    from serving_sampler_gb300 import _build
    import workloads

    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: a CUDA GPU is required for the native arm")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    _barrier(world)
    sv.load()

    w, meta = _listen(device, a.sessions)
    R, k = meta["R"], meta["k"]
    target, draft = w["target"], w["draft"]
    out = dict(accept_len=torch.empty(R, dtype=torch.int32, device=device),
               tokens=torch.empty(R, k + 1, dtype=torch.int32, device=device),
               branch=torch.empty(R, dtype=torch.int32, device=device),
               status=torch.empty(R, dtype=torch.int32, device=device))
    ws = torch.empty(sv.verify_greedy_workspace(R, k, 2, meta["V"]), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        sv.verify_greedy(target, R, k, 2, draft, out=out, workspace=ws, stream=stream)

    for _ in range(max(a.warmup, 3)):
        step()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        step()
    e1.record(stream)
    e1.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    clock_rows = clocks.stop()
    ms_local = e0.elapsed_time(e1) / a.steps
    ms = _max_over_ranks(ms_local, world, device)
    value = world * meta["logit_bytes"] / (ms * 1e-3) / 1e9
    rows_per_s = world * meta["rows"] / (ms * 1e-3)

    # end to end: pinned host inputs in, results out, every step
    e2e_steps = max(3, min(a.steps, 20))
    h_target = torch.empty(target.shape, dtype=target.dtype, pin_memory=True)
    h_target.copy_(target)
    h_draft = torch.empty(draft.shape, dtype=draft.dtype, pin_memory=True)
    h_draft.copy_(draft)
    h_out = {key: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for key, v in out.items()}
    d_target = torch.empty_like(target)
    d_draft = torch.empty_like(draft)

    def e2e_step():
        d_target.copy_(h_target, non_blocking=True)
        d_draft.copy_(h_draft, non_blocking=True)
        sv.verify_greedy(d_target, R, k, 2, d_draft, out=out, workspace=ws, stream=stream)
        for key, v in out.items():
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
    h2d = h_target.numel() * h_target.element_size() + h_draft.numel() * h_draft.element_size()
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    e2e_value = world * meta["logit_bytes"] / (e2e_ms * 1e-3) / 1e9
    del h_target, d_target

    peak, peak_kind = _peaks()
    achieved = meta["logit_bytes"] / (ms_local * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": _traffic_from_profile("greedy.cu"),
                "kernel": "argmax_segments_kernel<bf16> (+ greedy_finalize_kernel inside the same events)",
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        host = workloads.host_rows(target)
        gbs, rps, done, el = _oracle_sample(host, draft.cpu().numpy(), meta, a.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{done} sessions (65 rows x 151936 bf16 each) of the listen workload, {el:.1f} s, "
                         f"single-threaded fp64 C", "rows_per_s": rps}

    if rank == 0:
        line = {
            "metric": "verify logit GB/s (speculative-listening greedy verify, V=151936 bf16)",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"listen: {R} sessions x (32 main + 32 runner-up drafts) = 65 rows x 151936 "
                                   f"bf16 per session ({meta['logit_bytes'] / 1e9:.3f} GB of logits per step)",
                       "l2": f"inputs ({meta['logit_bytes'] / 1e9:.3f} GB) larger than L2 (129 MB); no flush",
                       "parallelism": f"replicas x{world}"},
            "rows_per_s": rows_per_s,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps},
            "gpu_launches": a.steps * sv.LAUNCHES["verify_greedy"],
            "clocks": Clocks.summarize(clock_rows),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    a = _args()
    if a.impl == "reference":
        return run_reference(a)
    return run_native(a)


if __name__ == "__main__":
    sys.exit(main())
