"""Benchmark of the verify step (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one verify round (plan + row pass + residual) over one synthetic
batch already resident in HBM.  value = verified logit rows (sum_r (k_r+1))
per second over all ranks; ranks run independent batches (weak scaling, no
collective on the data path).  The default workload, w4_v262144_bf16, is the
largest synthetic batch: 512 requests, k = 4, V = 262144, bf16 logits (2.4 GB
per step, far larger than the 129 MB L2, so no flush between steps).

The line also carries:
  roofline     achieved GB/s of the round = its algorithmic bytes B_alg / its
               CUDA-event time, against the measured HBM copy bandwidth.  B_alg is
               every logit row of the verified windows read once (2k+1 rows per
               sampling request, k+1 per greedy one) plus the small inputs and the
               outputs; re-reads for the correction draw are not counted.  Rows past
               a request's first rejection are never read, so the line also gives
               the bytes the round needed (positions 0..A) and, from the committed
               ncu capture, the DRAM bytes it actually moved;
  e2e          the same metric through specverify_run_host on pinned host inputs,
               outputs copied back, every step; the kernels read the pinned
               logits in place (only the rows a round reads cross the link);
  cpu_baseline the CPU oracle on a bounded sample of the same batch (1 core);
  clocks       SM clock samples taken during the timed region (NVML every
               millisecond, else nvidia-smi every 200 ms).
--impl reference times the CPU oracle instead (the only other arm there is).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified logit rows/sec"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "w4_v262144_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000
FLUSH_BYTES = 512 << 20


def truncated_draft_tokens(b, top_k: int, top_p: float, seed: int, chunk: int = 64):
    """Input preparation for truncated rounds: the draft tokens of sampling
    requests are redrawn from their truncated draft distributions (plain torch
    ops: temperature, then top-k, then top-p on the survivors), as a drafter
    sampling from its truncated distribution would emit them."""
    import torch
    dev = b.draft.device
    gen = torch.Generator(device=dev).manual_seed(seed)
    nd = b.num_draft.cpu().numpy()
    temps = b.temperature.cpu().numpy()
    row_t = torch.as_tensor(np.repeat(temps, nd), dtype=torch.float32, device=dev)
    V = b.draft.shape[1]
    for s0 in range(0, b.total_draft, chunk):
        T = row_t[s0:s0 + chunk]
        x = b.draft[s0:s0 + chunk].float() / torch.where(T > 0, T, 1.0)[:, None]
        if 0 < top_k < V:
            kth = torch.topk(x, top_k, dim=1).values[:, -1:]
            x = torch.where(x >= kth, x, float("-inf"))
        if top_p < 1.0:
            srt, _ = torch.sort(x, dim=1, descending=True)
            p = torch.softmax(srt, dim=1)
            above = torch.cumsum(p, dim=1) - p          # mass of the larger survivors
            keep = above < top_p
            thr = torch.where(keep, srt, float("inf")).min(dim=1, keepdim=True).values
            x = torch.where(x >= thr, x, float("-inf"))
        tok = torch.multinomial(torch.softmax(x, dim=1), 1, generator=gen).squeeze(1)
        b.tokens[s0:s0 + chunk] = torch.where(T > 0, tok.to(torch.int32), b.tokens[s0:s0 + chunk])

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="requests in the oracle sample (0 = about 10 s of work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--host-reads", default="auto", choices=["auto", "stage"],
                    help="e2e: read pinned host logits in place (auto) or copy them in (stage)")
    ap.add_argument("--schedule", default="auto", choices=["auto", "waves"],
                    help="launch layout of a round (results do not depend on it)")
    ap.add_argument("--depth", type=int, default=0,
                    help="positions per wave launch (0 = chosen per run)")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per batch (0 = the workload's own); for profiling captures")
    ap.add_argument("--top-k", type=int, default=None,
                    help="truncate every target and draft row to its top-k logits")
    ap.add_argument("--top-p", type=float, default=None,
                    help="truncate every target and draft row to its top-p nucleus")
    ap.add_argument("--trunc-path", choices=["masked", "copy"], default="masked",
                    help="truncation: thresholds and a mask on load inside the round "
                         "(specverify_run_truncated), or a truncated copy then the round")
    ap.add_argument("--trim", type=float, default=None,
                    help="verify windows trimmed from draft confidences, at this cost per "
                         "verified position (specverify_run_trimmed)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the slowest rank's time sets a weak-scaling
    step); x itself when there is one rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_sec(rows_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of a weak-scaling step: every rank verifies its own
    batch of rows_per_rank rows; the step ends when the slowest rank does."""
    return world * rows_per_rank / (ms_max * 1e-3)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources a verify round on the default schedule is built from: the plan
# and wave kernels, their device helpers, and the host code that launches them.
ROUND_SOURCES = ("sv_device.cuh", "sv_kernels.cuh", "specverify.cu")


def _code_only(text: str) -> str:
    """C++ source without comments and blank space, so that an edit to a comment
    leaves the hash of the code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":  # a literal, copied as it is
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_10_gb300", "csrc")
    for name in ROUND_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update((name + "\n" + _code_only(f.read())).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per round from the committed ncu summary, if it was taken on
    the current sources of the round's kernels; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class NvmlClocks:
    """Read-only NVML queries through ctypes (libnvidia-ml): the SM clock, its
    maximum and the clock event reasons of one GPU, polled every millisecond
    from a host thread between mark("start") and mark("stop").  None of the
    calls changes a setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index),
                                                  ctypes.byref(self.dev)) != 0:
            raise RuntimeError("no NVML handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.running = False

    def _one(self):
        ct = self.ct
        mhz, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(mhz)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ct.byref(mx))
        self.reasons_fn(self.dev, ct.byref(rs))
        return mhz.value, mx.value, rs.value

    def _loop(self):
        while self.running:
            one = self._one()
            if one is not None:
                self.samples.append(one)
            time.sleep(0.001)

    def start(self):
        self.samples = []
        self.running = True
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.running = False
        self.thread.join(timeout=1.0)
        if not self.samples:
            return None
        reasons = sorted({name for _, _, r in self.samples
                          for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(s for s, _, _ in self.samples),
                "sm_max_mhz": max(m for _, m, _ in self.samples), "reasons": reasons,
                "samples": len(self.samples), "window": "timed region (NVML, 1 ms period)"}


class ClockSampler:
    """Clock samples of the timed region: NVML polled every millisecond when the
    library loads, else nvidia-smi every 200 ms (samples inside [start, stop])."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t_start = self.t_stop = None
        try:
            self.nvml = NvmlClocks(gpu_index)
        except Exception:
            self.nvml = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())
        if self.nvml is not None:
            if which == "start":
                self.nvml.start()
            elif which == "stop":
                self.nvml_info = self.nvml.stop()

    def stop(self):
        fast = getattr(self, "nvml_info", None)
        if fast is not None:
            if self.proc is not None:
                self.proc.terminate()
                try:
                    self.proc.wait(timeout=5)
                except Exception:
                    self.proc.kill()
            return fast
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [s for t, s in self.samples if self.t_start <= t <= self.t_stop + 0.2]
        window = "timed region"
        if not inside:
            inside = [s for _, s in self.samples][-3:]
            window = "nearest samples (timed region shorter than the sampling period)"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            parts = [p.strip() for p in s.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


def oracle_rows_per_sec(batch, requests, full=False):
    """Time the CPU oracle on the given requests of `batch` (single thread).
    With full=True (requests = the whole batch) also return the oracle's
    outputs and the inputs it was given."""
    import oracle
    from speculative_decoding_verification_10_gb300 import workloads as W
    inp = (batch if full else W.subset(batch, requests)).numpy_inputs()
    t0 = time.perf_counter()
    out = oracle.verify(inp["target"], inp["draft"], inp["tokens"], inp["num_draft"],
                        inp["temperature"], 1, inp["max_k"], request_ids=inp["request_ids"])
    dt = time.perf_counter() - t0
    rows = int(inp["num_draft"].astype(np.int64).sum()) + len(requests)
    if full:
        return rows / dt, dt, rows, out, inp
    return rows / dt, dt, rows


def cpu_model():
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in outp.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def bench_parity(v, b, oracle_out, inp):
    """The benchmark batch verified once more (seed 1, debug outputs) and compared
    with the oracle request by request, outside the timed region.  Counts the
    requests checked, the exact ones and the near-threshold exemptions."""
    import torch
    from tests import parity
    res = v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, 1, debug=True)
    torch.cuda.synchronize()
    gpu = {"accepted_len": res.accepted_len.cpu().numpy(), "committed": res.committed.cpu().numpy(),
           "flags": res.flags.cpu().numpy(), "p_y": res.p_y.cpu().numpy(),
           "q_y": res.q_y.cpu().numpy(), "u": res.u.cpu().numpy(),
           "req_status": res.req_status.cpu().numpy(), "status": v.status()}
    rep = parity.compare(gpu, oracle_out, inp, 1)
    exempt = rep["exempt_accept"] + rep["exempt_race"] + rep["exempt_residual_mass"]
    return {"requests_checked": rep["requests"], "exact": rep["requests"] - exempt,
            "exempt_accept": rep["exempt_accept"], "exempt_race": rep["exempt_race"],
            "exempt_residual_mass": rep["exempt_residual_mass"],
            "seed": 1, "rule": "tokens, lengths and flags bit-exact; decisions within 1e-5 "
                               "relative of their threshold exempt and counted"}


def estimate_sample(batch, target_seconds=15.0):
    """Requests whose oracle run takes about target_seconds (from a 1-request probe)."""
    _, dt, _ = oracle_rows_per_sec(batch, [0])
    n = int(max(1, min(batch.batch, target_seconds / max(dt, 1e-4))))
    return n


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import torch
    from speculative_decoding_verification_10_gb300 import workloads as W
    dev = f"cuda:{local}" if torch.cuda.is_available() else "cpu"
    b = W.make_batch(args.workload, device=dev)
    # the whole batch per step when the run fits in about five minutes (it does
    # for twenty steps and five warm-up steps), else a bounded sample of it
    per_step = args.cpu_sample or max(1, min(b.batch, int(300.0 / max(1, args.steps + args.warmup)
                                                        / max(_probe_seconds(b), 1e-4))))
    times, rows_total = [], 0
    order = np.arange(b.batch)
    for s in range(args.warmup + args.steps):
        start = (s * per_step) % b.batch
        req = np.sort(order[(start + np.arange(per_step)) % b.batch])
        rps, dt, rows = oracle_rows_per_sec(b, req)
        if s >= args.warmup:
            times.append(dt)
            rows_total += rows
    value = rows_total / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": b.batch, "k": W.SPECS[args.workload].k,
                       "vocab": b.vocab, "logits": b.dtype,
                       "rows_per_step": rows_total // max(1, args.steps)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": (f"the whole batch ({b.batch} requests) per step"
                                        if per_step == b.batch else
                                        f"{per_step} of {b.batch} requests of {args.workload} "
                                        "per step")},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _probe_seconds(b):
    """Oracle seconds per request, from the first few requests."""
    n = min(4, b.batch)
    _, dt, _ = oracle_rows_per_sec(b, np.arange(n))
    return dt / n


def measure_e2e(args, b, v, world, dev):
    """rows/s through specverify_run_host: pinned host inputs in, outputs out, per step."""
    import torch
    import torch.distributed as dist
    hb = b.to("cpu")
    h_target = hb.target.pin_memory()
    h_draft = hb.draft.pin_memory()
    h_tokens, h_nd, h_temp = hb.tokens.pin_memory(), hb.num_draft.pin_memory(), hb.temperature.pin_memory()
    h_acc = torch.empty(b.batch, dtype=torch.int32).pin_memory()
    h_com = torch.empty(b.batch, b.max_k + 1, dtype=torch.int32).pin_memory()
    h_flg = torch.empty(b.total_draft, dtype=torch.uint8).pin_memory()
    for _ in range(2):
        v.run_host(h_target, h_draft, h_tokens, h_nd, h_temp, 1, h_acc, h_com, h_flg)
    if world > 1:
        dist.barrier()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        v.run_host(h_target, h_draft, h_tokens, h_nd, h_temp, 1, h_acc, h_com, h_flg)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_t = torch.tensor([e2e_s], device=dev)
    if world > 1:
        dist.all_reduce(e2e_t, op=dist.ReduceOp.MAX)
    e2e_s = float(e2e_t.item())
    small = 4 * (h_tokens.numel() + h_nd.numel() + h_temp.numel())
    in_place = v.last_host_reads() == 1
    if in_place:
        # the kernels read the rows of every wave a request takes part in where
        # they lie; the waves copy each sampled row to the device as it
        # streams, so a correction draw reads its two rows from there
        depth = v.wave_depth(b.batch)
        A = h_acc.numpy().astype(np.int64)
        k = h_nd.numpy().astype(np.int64)
        sampling = h_temp.numpy() > 0
        last = np.minimum(k, (A // depth + 1) * depth - 1)
        rows = np.where(sampling, 2 * np.minimum(last + 1, k) + (last == k),
                        last + 1)
        logits = int(rows.sum()) * b.vocab * h_target.element_size()
    else:
        logits = h_target.numel() * h_target.element_size() + h_draft.numel() * h_draft.element_size()
    h2d = logits + small
    d2h = 4 * h_acc.numel() + 4 * h_com.numel() + h_flg.numel()
    return {"value": world * b.verified_rows() / e2e_s, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
            "logits": ("pinned host rows read in place by the kernels (only the rows a round "
                       "reads cross the link)" if in_place else
                       "whole window copied host to device each step")}



def run_ours(args):
    import torch
    import torch.distributed as dist
    from speculative_decoding_verification_10_gb300 import Verifier, build
    from speculative_decoding_verification_10_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()

    spec = W.SPECS[args.workload]
    b = W.make_batch(args.workload, device=dev, gen_seed=spec.gen_seed + 7919 * rank,
                     batch=args.batch or None)
    torch.cuda.empty_cache()
    rows_per_step = b.verified_rows()
    es = 2 if b.dtype == "bf16" else 4
    k = b.num_draft.cpu().numpy().astype(np.int64)
    t = b.temperature.cpu().numpy()
    full_window_bytes = b.full_window_bytes()

    v = Verifier(b.batch, b.max_k, b.vocab, b.dtype, device=local, host_staging=not args.no_e2e)
    v.set_schedule(args.schedule)
    v.set_depth(args.depth)
    v.set_host_reads(args.host_reads)
    out = v.outputs(b.batch, b.total_draft)
    stream = torch.cuda.current_stream(dev)

    conf = cost = None
    if args.trim is not None:
        # synthetic draft confidences: c_i uniform in [0.6, 1) from a seeded generator
        gconf = torch.Generator("cpu").manual_seed(4242 + rank)
        conf = (0.6 + 0.4 * torch.rand(b.total_draft, generator=gconf)).to(dev)
        cost = torch.full((b.batch,), float(args.trim), dtype=torch.float32, device=dev)

    trunc = None
    if args.top_k is not None or args.top_p is not None:
        from speculative_decoding_verification_10_gb300 import truncate
        tk = torch.full((b.batch,), int(args.top_k or 0), dtype=torch.int32, device=dev)
        tp = torch.full((b.batch,), float(args.top_p if args.top_p is not None else 1.0),
                        dtype=torch.float32, device=dev)
        truncated_draft_tokens(b, int(args.top_k or 0),
                               float(args.top_p if args.top_p is not None else 1.0), 4343 + rank)
        if args.trunc_path == "copy":
            tgt_out, drf_out = torch.empty_like(b.target), torch.empty_like(b.draft)
            trunc = (truncate, tk, tp, tgt_out, drf_out)
        else:
            trunc = (None, tk, tp, None, None)

    def step():
        if trunc is not None:
            fn, tk, tp, to, do = trunc
            if fn is None:
                # thresholds, then the round masking the rows as it loads them
                return v.run_truncated(b.target, b.draft, b.tokens, b.num_draft, b.temperature,
                                       tk, tp, 1, out=out)
            fn(b.target, b.draft, b.num_draft, b.temperature, tk, tp, out_target=to,
               out_draft=do)
            v.run(to, do, b.tokens, b.num_draft, b.temperature, 1, out=out)
            return out
        if conf is not None:
            return v.run_trimmed(b.target, b.draft, b.tokens, b.num_draft, conf, cost,
                                 b.temperature, 1)
        v.run(b.target, b.draft, b.tokens, b.num_draft, b.temperature, 1, out=out)
        return out

    for _ in range(max(3, args.warmup)):
        res = step()
    torch.cuda.synchronize()
    if v.status() != 0:
        raise RuntimeError(f"verify status {v.status()} on the benchmark batch")
    # bytes the round must read: positions 0..A of each request (target and draft
    # rows when sampling, target rows when greedy) and the bonus row when A = k
    # (k = the verified window: the trimmed one in a trimmed round)
    A = res.accepted_len.cpu().numpy().astype(np.int64)
    if conf is not None:
        k = res.verified_k.cpu().numpy().astype(np.int64)
        rows_per_step = int((k + 1).sum())
    rows_needed = np.where(t > 0, np.where(A < k, 2 * (A + 1), 2 * k + 1), A + 1)
    needed_bytes = int(rows_needed.sum()) * b.vocab * es
    # B_alg: every row of the verified windows once, plus inputs and outputs
    window_rows = np.where(t > 0, 2 * k + 1, k + 1)
    window_bytes = int(window_rows.sum()) * b.vocab * es
    alg_bytes = window_bytes + b.io_bytes()

    trunc_ms = None
    if trunc is not None and trunc[0] is not None:
        # the truncation pass alone (it reads every window row and writes it once)
        fn, tk, tp, to, do = trunc
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(20):
            fn(b.target, b.draft, b.num_draft, b.temperature, tk, tp, out_target=to, out_draft=do)
        e1.record(stream)
        torch.cuda.synchronize()
        trunc_ms = e0.elapsed_time(e1) / 20

    # A step whose window is below twice the L2 would find last step's rows
    # there: such steps get an L2 eviction before each round (one buffer
    # written, then another read, so no dirty lines drain inside the round),
    # and each round is timed alone on its own events.
    flush = window_bytes < 2 * L2_BYTES
    if flush:
        fl_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        fl_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        fl_sink = torch.empty((), dtype=torch.float32, device=dev)

        def evict_l2():
            fl_w.fill_(0.0)
            torch.sum(fl_r, dim=0, out=fl_sink)
    n_ev = args.steps if flush else min(64, args.steps)
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for e in ev_s + ev_e:        # torch creates the CUDA event on first record
        e.record(stream)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)

    # timed region: K steps, CUDA events on the launching stream
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("start")
    t_start.record(stream)
    # the launches of each of the first n_ev timed rounds are bracketed by events
    if flush:
        for i in range(args.steps):
            evict_l2()
            v.set_timing_events(ev_s[i:i + 1], ev_e[i:i + 1])
            step()
    else:
        v.set_timing_events(ev_s, ev_e)
        for i in range(args.steps):
            if i == n_ev:
                v.set_timing_events([], [])
            step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    clocks.mark("stop")
    kernel_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(n_ev)]
    v.set_timing_events([], [])
    if world > 1:
        dist.barrier()
    # with evictions the step time is the rounds' own, summed; else the region's
    ms = (sum(kernel_ms) if flush else t_start.elapsed_time(t_stop)) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    clock_info = clocks.stop()

    # end to end through the host-buffer entry point (pinned host inputs)
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, b, v, world, dev)

    # CPU oracle baseline on a bounded sample (rank 0, N = 1 only); when the
    # sample is the whole batch, the oracle's outputs also check the GPU's
    # outputs for the same batch request by request (the parity record)
    cpu = None
    par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = args.cpu_sample or estimate_sample(b)
        if n >= b.batch and conf is None and trunc is None:
            rps, dt, rows, orc, inp = oracle_rows_per_sec(b, np.arange(b.batch), full=True)
            par = bench_parity(v, b, orc, inp)
        else:
            req = np.sort(np.random.default_rng(0).choice(b.batch, size=n, replace=False))
            rps, dt, rows = oracle_rows_per_sec(b, req)
        cpu = {"value": rps, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"{n if n < b.batch else b.batch} of {b.batch} requests "
                         f"({rows} verified rows), {dt:.1f} s"}

    if rank != 0:
        v.close()
        if world > 1:
            dist.destroy_process_group()
        return 0

    kernel_avg_ms = float(np.mean(kernel_ms))
    peak, peak_kind = measured_peak()
    achieved = alg_bytes / (kernel_avg_ms * 1e-3) / 1e9
    needed_gbs = needed_bytes / (kernel_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload) if conf is None and trunc is None else None
    line = {
        "metric": METRIC, "value": job_rows_per_sec(rows_per_step, world, ms_max), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "batch": b.batch, "k": spec.k,
                   "vocab": b.vocab, "logits": b.dtype, "rows_per_step": rows_per_step,
                   "alg_bytes_per_step": alg_bytes,
                   "step_gbs": alg_bytes / (ms_max * 1e-3) / 1e9,
                   "rows_needed_per_step": int(rows_needed.sum()),
                   "window_rows_per_step": int(window_rows.sum()),
                   "mean_accepted": float(A.mean()),
                   "l2": (("L2 evicted before every round (%d MB written, then %d MB read; "
                           "rounds timed alone): the %.3f GB window is below twice the 129 MB L2")
                          % (FLUSH_BYTES >> 20, FLUSH_BYTES >> 20, window_bytes / 1e9)
                          if flush else
                          "no flush: each step reads %.2f GB of a %.2f GB window, larger than "
                          "the 129 MB L2" % (needed_bytes / 1e9, window_bytes / 1e9)),
                   "parallelism": f"replicas x{world}",
                   "schedule": args.schedule, "depth": args.depth,
                   "trim_cost": args.trim, "top_k": args.top_k, "top_p": args.top_p,
                   "truncation": (None if trunc is None else
                                  ("copy: the truncated rows written, then the round"
                                   if trunc[0] is not None else
                                   "masked: a threshold pass, then the round masking rows "
                                   "on load (both inside the timed round)")),
                   "truncation_bytes_per_step": (0 if trunc is None else
                                                 (2 if trunc[0] is not None else 1)
                                                 * full_window_bytes),
                   "truncation_ms": trunc_ms,
                   "truncation_gbs": (2 * full_window_bytes / (trunc_ms * 1e-3) / 1e9
                                      if trunc_ms else None)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "sv_wave", "kernel_ms": kernel_avg_ms,
                     "window": "one round: sv_plan + its sv_wave launches, back to back",
                     "alg_bytes_per_launch": alg_bytes,
                     "needed_bytes_per_launch": needed_bytes,
                     "needed_gbs": needed_gbs, "needed_frac": needed_gbs / peak,
                     "dram_gbs": (traffic / (kernel_avg_ms * 1e-3) / 1e9
                                  if traffic is not None else None),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback"},
        "cpu_baseline": cpu,
        "parity": par,
        "e2e": e2e,
        "clocks": clock_info,
        "gpu_launches": v.launches_per_run(b.batch) * args.steps,
    }
    print(json.dumps(line), flush=True)
    v.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_tree(args):
    """Greedy tree verification rounds (specverify_tree_run) on a synthetic tree batch."""
    import torch
    import torch.distributed as dist
    from speculative_decoding_verification_10_gb300 import TreeVerifier, build
    from speculative_decoding_verification_10_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    tb = W.make_tree_batch(args.workload, device=dev, batch=args.batch or None)
    tv = TreeVerifier(tb.batch, tb.max_nodes, tb.vocab, tb.dtype, device=local)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        res = tv.run(tb.target, tb.num_nodes, tb.parent, tb.tokens)
    torch.cuda.synchronize()
    if tv.status() != 0:
        raise RuntimeError(f"tree status {tv.status()}")
    A = res.accepted_len.cpu().numpy()
    # the walk reads A_r + 1 rows per tree; when those fit twice in the L2,
    # every round runs after an L2 eviction and is timed alone
    walked = int((A.astype(np.int64) + 1).sum()) * tb.row_bytes()
    flush = walked < 2 * L2_BYTES
    if flush:
        fl_w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        fl_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        fl_sink = torch.empty((), dtype=torch.float32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps if flush else 1)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("start")
    t0.record(stream)
    for i in range(args.steps):
        if flush:
            fl_w.fill_(0.0)
            torch.sum(fl_r, dim=0, out=fl_sink)
            ev[i][0].record(stream)
        tv.run(tb.target, tb.num_nodes, tb.parent, tb.tokens)
        if flush:
            ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("stop")
    ms = (sum(a.elapsed_time(b) for a, b in ev) if flush else t0.elapsed_time(t1)) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    clock_info = clocks.stop()
    # end to end through the public API: pinned host inputs copied in, outputs back
    h = [x.cpu().pin_memory() for x in (tb.target, tb.num_nodes, tb.parent, tb.tokens)]
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    torch.cuda.synchronize()
    te = time.perf_counter()
    for _ in range(e2e_steps):
        d = [x.to(dev, non_blocking=True) for x in h]
        r2 = tv.run(*d)
        out_host = (r2.accepted_len.cpu(), r2.path.cpu(), r2.committed.cpu())
    e2e_s = (time.perf_counter() - te) / e2e_steps
    rows = tb.rows()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = tb.batch
        sub = slice(0, n * (tb.max_nodes + 1))
        tgt = tb.target[sub].cpu()
        tgt = tgt.view(torch.int16).numpy().view(np.uint16) if tb.dtype == "bf16" else tgt.numpy()
        tc = time.perf_counter()
        oracle.tree_greedy(tgt, tb.num_nodes[:n].cpu().numpy(),
                           tb.parent[:n * tb.max_nodes].cpu().numpy(),
                           tb.tokens[:n * tb.max_nodes].cpu().numpy(), tb.max_nodes)
        dt = time.perf_counter() - tc
        cpu = {"value": n * (tb.max_nodes + 1) / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} of {tb.batch} trees ({n * (tb.max_nodes + 1)} rows), {dt:.1f} s"}
    tv.close()
    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    alg = rows * tb.row_bytes()
    achieved = alg / (ms_max * 1e-3) / 1e9
    h2d = sum(x.numel() * x.element_size() for x in h)
    d2h = sum(x.numel() * x.element_size() for x in out_host)
    line = {
        "metric": METRIC, "value": job_rows_per_sec(rows, world, ms_max), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": tb.batch, "nodes": tb.max_nodes,
                   "vocab": tb.vocab, "logits": tb.dtype, "rows_per_step": rows,
                   "mean_accepted": float(A.mean()),
                   "l2": (("L2 evicted before every round (%d MB written, then %d MB read; "
                           "rounds timed alone): a round walks %.1f MB of a %.2f GB tree window"
                           % (FLUSH_BYTES >> 20, FLUSH_BYTES >> 20, walked / 1e6, alg / 1e9))
                          if flush else
                          "no flush: each round walks %.2f GB, more than twice the 129 MB L2"
                          % (walked / 1e9)),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "sv_tree_path", "alg_bytes_per_launch": alg,
                     "walked_bytes_per_launch": walked,
                     "walked_gbs": walked / (ms_max * 1e-3) / 1e9,
                     "window": "one round: sv_tree_plan + sv_tree_path",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * rows / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "clocks": clock_info,
        "gpu_launches": 2 * args.steps,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    from speculative_decoding_verification_10_gb300 import workloads as W
    if args.workload in W.TREE_SPECS:
        return run_tree(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
