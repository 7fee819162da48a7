"""Benchmark of one DSpark draft-head round (draft -> schedule -> verify) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl dspark|reference]

A step is one whole round over one batch: base logits (LM head), the gamma-step
Markov/confidence loop, the prefix scheduler and verification.  Inputs are
synthetic, seeded, and resident in HBM before the timed region; the LM head
weight (1.85 GB at the default workload) is larger than L2, so successive steps
do not run from cache.  With N > 1 (launched by torchrun) every rank runs an
independent replica on its own GPU: there is no collective on the data path.

Prints one JSON line (rank 0).  `value` is drafted tokens/s over all ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "drafted tokens/s"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "v4_dspark5"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    # ~1 s of timed rounds at V4, so the clock sampler (20 ms) sees it many times
    p.add_argument("--steps", type=int, default=600)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--impl", default="dspark", choices=["dspark", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--fused-variant", action="store_true",
                   help="also time the fused single-contraction draft step (a measured "
                        "variant; the main line is unchanged)")
    p.add_argument("--rnn-variant", action="store_true",
                   help="also time the RNN-head draft (a measured variant) against the loop")
    p.add_argument("--sts-fit", action="store_true",
                   help="also time one STS fit over 1M synthetic held-out rounds")
    p.add_argument("--cpu-sample", type=int, default=0,
                   help="requests in the CPU-oracle sample (0 = sized automatically)")
    return p.parse_args()


# --------------------------------------------------------------- helpers ----

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """Slowest rank's time: the whole job finishes when the last replica does."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if (torch.cuda.is_available() and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, ms_per_step_max: float, ws: int) -> float:
    """Units processed by all replicas per second of the slowest replica's step."""
    return ws * units_per_rank / (ms_per_step_max * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return dict(hbm_gbs=j["hbm_gbs"], bf16=j["bf16_tflops"],
                    bf16_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from before the
    warm-up on; stop() keeps the samples stamped inside the timed region (the
    one nearest its middle when the region is shorter than the period)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def region(self, t0, t1):
        """Host wall-clock bounds (datetime) of the timed region."""
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(f[2]), float(f[3]),
                             {n for n, v in zip(names, f[6:10]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        if not rows:
            return None
        inside = rows
        if self.t0 is not None:
            inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
            if not inside:
                mid = self.t0 + (self.t1 - self.t0) / 2
                inside = [min(rows, key=lambda r: abs((r[0] - mid).total_seconds()))]
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(set().union(*(r[3] for r in inside))),
                "samples": len(inside),
                "window_ms": None if self.t0 is None else
                round((self.t1 - self.t0).total_seconds() * 1e3, 1)}


# Sources that define the LM-head kernel; a profile taken on other sources is stale.
LM_HEAD_SOURCES = ["lm_head.cu", "umma_gemm_pair.cuh", "umma_gemm.cuh", "umma_skinny.cuh",
                   "tcgen05.cuh", "common.cuh"]


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        p = os.path.join(ROOT, "speculative_decoding_draft_02_gb300", "csrc", n)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, src_hash: str, units: float, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel and on this workload (else None).  The
    summary states the bytes of its captured launch and the units it processed;
    scaled by `units`."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith(" "):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_hash") != src_hash or kv.get("workload", "").split()[:1] != [workload]:
        return None
    try:  # "units_per_launch: 1280  (what they are)"
        b = float(kv["dram_bytes_per_launch"].split()[0])
        u = float(str(kv.get("units_per_launch", units)).split()[0])
    except (KeyError, ValueError, IndexError):
        return None
    return b * units / u


# ----------------------------------------------------------- workload -----

def replica_seed(w, rank: int) -> int:
    """Each replica draws its own batch (independent requests per GPU)."""
    return w.seed + 1000 * rank


def build_inputs(w, rank: int, device="cuda"):
    inp = workloads.make_inputs(w, device=device, seed=replica_seed(w, rank))
    # Synthetic target model: target logits = draft base logits + N(0, sigma_r)
    # for positions 1..gamma, and a fresh hidden state through the shared head
    # for position gamma + 1.  Built with cuBLAS (torch.matmul) once, untimed.
    R, G, V, d = w.R, w.gamma, w.V, w.d
    Wl = inp["W_lm"].to(torch.bfloat16)
    base = torch.matmul(inp["h"].to(torch.bfloat16).reshape(R * G, d), Wl.t()).view(R, G, V)
    nxt = torch.matmul(inp["h_next"].to(torch.bfloat16), Wl.t()).view(R, 1, V)
    target = torch.cat([base, nxt], dim=1).float().add_(inp.pop("noise").float())
    inp["target"] = target.to(torch.bfloat16).contiguous()
    del base, nxt, target
    torch.cuda.empty_cache()
    return inp


# ------------------------------------------------------- CPU baseline -----

def cpu_oracle_round(w, inp_cpu, S: int):
    """Run the oracle's full round on the first S requests; returns seconds."""
    import oracle
    R, G, V, d = w.R, w.gamma, w.V, w.d
    t0 = time.perf_counter()
    h = inp_cpu["h"][:S]
    base = oracle.base_logits(h.reshape(S * G, d), inp_cpu["W_lm"], vocab_chunk=8192).reshape(
        S, G, V)
    dr = oracle.markov_draft(base, h, inp_cpu["anchor"][:S], inp_cpu["W1"], inp_cpu["W2"],
                             inp_cpu["w_conf"], inp_cpu["T"], w.tau, inp_cpu["draft_seed"],
                             keep_logits=w.tau > 0)
    sps = inp_cpu["sps"]
    sch = oracle.schedule(dr["conf"].astype(np.float32), sps, oracle.UNCONSTRAINED)
    oracle.verify(dr["tokens"], sch["len"], dr.get("logits"), inp_cpu["target"][:S], w.tau,
                  inp_cpu["verify_seed"])
    return time.perf_counter() - t0


def cpu_inputs(w, inp_gpu):
    keys = ["h", "anchor", "W_lm", "W1", "W2", "w_conf", "T", "sps"]
    out = {k: inp_gpu[k].cpu() for k in keys}
    out["draft_seed"] = inp_gpu["draft_seed"]
    out["verify_seed"] = inp_gpu["verify_seed"]
    return out


def sample_size(w, cpu, target, avail: int, target_s: float) -> int:
    """Requests whose oracle round takes about target_s seconds, from the
    marginal cost per request between a 1- and a 4-request probe (a round has
    a fixed part that one probe alone would charge to its single request)."""
    cpu["target"] = target[:4].cpu()
    t1 = cpu_oracle_round(w, cpu, 1)
    t4 = cpu_oracle_round(w, cpu, min(4, avail))
    per = max((t4 - t1) / 3.0, 1e-4)
    fixed = max(t1 - per, 0.0)
    return int(max(1, min(avail, math.floor((target_s - fixed) / per))))


def cpu_baseline(w, inp_gpu, S: int, target_s: float = 15.0):
    cpu = cpu_inputs(w, inp_gpu)
    cores = torch.get_num_threads()
    if not S:
        S = sample_size(w, cpu, inp_gpu["target"], w.R, target_s)
    cpu["target"] = inp_gpu["target"][:S].cpu()
    t = cpu_oracle_round(w, cpu, S)
    return {"value": S * w.gamma / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one full round (LM head, {w.gamma}-step Markov loop, schedule, verify) "
                      f"for the first {S} of {w.R} requests of {w.name}, float64 numpy, "
                      f"{t:.1f} s on {os.cpu_count()} host cores"}


# ------------------------------------------------------------ arms --------

def run_reference(args, w, ws, rank):
    """The CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    torch.manual_seed(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        inp = build_inputs(w, 0)
    else:
        small = w.with_(R=min(w.R, 4))
        inp = workloads.make_inputs(small, device="cpu")
        inp["target"] = torch.zeros((small.R, w.gamma + 1, w.V), dtype=torch.bfloat16)
    cpu = cpu_inputs(w, inp)
    # size one step so that warmup + steps fit in about three minutes
    S = args.cpu_sample or 1
    avail = int(inp["h"].shape[0])  # requests built (all of them when CUDA builds the inputs)
    if not args.cpu_sample:
        S = sample_size(w, cpu, inp["target"], avail, 180.0 / (args.steps + args.warmup))
    S = min(S, avail)
    cpu["target"] = inp["target"][:S].cpu()
    for _ in range(args.warmup):
        cpu_oracle_round(w, cpu, S)
    times = [cpu_oracle_round(w, cpu, S) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    value = S * w.gamma / sec
    cores = torch.get_num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "gamma": w.gamma, "V": w.V, "r": w.r, "d": w.d,
                   "tau": w.tau, "sample_requests": S},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: one oracle round for {S} of {w.R} requests"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_dspark(args, w, ws, rank, local):
    import speculative_decoding_draft_02_gb300 as dsp
    from speculative_decoding_draft_02_gb300 import build as dsp_build
    if rank == 0:
        dsp_build.build()
    barrier(ws)
    dsp.load_library()
    inp = build_inputs(w, rank)
    R, G, V, r, d = w.R, w.gamma, w.V, w.r, w.d
    head = dsp.DraftHead.from_weights(R, G, inp["W_lm"], inp["W1"], inp["W2"], inp["w_conf"],
                                      inp["T"])
    rnd = dsp.Round(head)
    h = inp["h"].to(torch.bfloat16).reshape(R * G, d).contiguous()
    anchor = inp["anchor"].contiguous()
    target = inp["target"]
    sps = inp["sps"].contiguous()
    tau, ds, vs = w.tau, inp["draft_seed"], inp["verify_seed"]
    stream = torch.cuda.current_stream()
    dims = head.dims

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsp.dspark_lm_head(dims, h, head.W_lm, rnd.base)
        if ev is not None:
            ev[1].record(stream)
        dsp.dspark_markov_draft(dims, rnd.base, h, anchor, head.W1, head.W2t, head.w_conf,
                                head.T, tau, ds, rnd.tokens, rnd.conf, rnd.logp_d, rnd.lse_d,
                                rnd.ws_draft)
        if ev is not None:
            ev[2].record(stream)
        rnd.schedule(sps)
        if ev is not None:
            ev[3].record(stream)
        rnd.verify(anchor, target, tau, vs)
        if ev is not None:
            ev[4].record(stream)

    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    dsp.check_device_status()

    # timed region: K whole rounds, events around each stage on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    n0 = dsp.dspark_launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # NVTX range "timed": a profiler can capture exactly the timed rounds
    torch.cuda.nvtx.range_push("timed")
    t_host0 = datetime.datetime.now()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_host1 = datetime.datetime.now()
    barrier(ws)
    launches = dsp.dspark_launch_count() - n0
    if clocks:
        clocks.region(t_host0, t_host1)
    clk = clocks.stop() if clocks else None
    ms = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms, ws)
    stage = {k: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
             for i, k in enumerate(["lm_head", "markov_loop", "schedule", "verify"])}
    dsp.check_device_status()
    K_adm = int(rnd.K.item())
    acc = rnd.accepted.float().mean().item()

    # roofline of the dominant kernel (the LM-head GEMM, tensor-bound); a kernel
    # timed inside a long loop runs under the power cap: the sustained peak
    peaks = measured_peaks()
    long_run = ms * args.steps >= 500.0 and peaks["bf16_sustained"]
    tc_peak = peaks["bf16_sustained"] if long_run else peaks["bf16"]
    tc_kind = ("sustained bf16 (timed inside a loop of %.1f s)" % (ms * args.steps / 1e3)
               if long_run else "burst bf16")
    ridge = tc_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)  # FLOP per byte where the bounds meet

    def roofline(flops, nbytes, t_ms):
        """Against the tensor peak above the ridge, against HBM below it."""
        if flops / nbytes >= ridge:
            ach = flops / (t_ms * 1e-3) / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": ach / tc_peak, "peak_source": peaks["source"] + " " + tc_kind}
        ach = nbytes / (t_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_source": peaks["source"] + " copy"}

    # LM head: 2 M V d FLOP over W_lm, h and the base logits (M = R gamma rows)
    lm_roof = roofline(2.0 * R * G * V * d, 2.0 * (V * d + R * G * d + R * G * V), stage["lm_head"])
    src = kernel_source_hash(LM_HEAD_SOURCES)
    lm_roof.update({"traffic": profiled_traffic("lm_head", src, R * G, w.name),
                    "kernel": "lm_head"})
    # the Markov loop: per step W2t, the base-logit rows and E; 2 R r V FLOP
    markov_bytes = G * (V * r * 2 + R * V * 2 + R * r * 2)
    markov_roof = roofline(G * 2.0 * R * r * V, markov_bytes, stage["markov_loop"])
    markov_gbs = markov_bytes / (stage["markov_loop"] * 1e-3) / 1e9
    # verify against HBM over the rows it reads (the round's own lengths)
    ln = rnd.len.long().cpu()
    acc_n = rnd.accepted.long().cpu()
    row = V * 2
    if w.tau > 0:
        rejected = acc_n < ln
        vbytes = int(ln.sum()) * row                   # target rows 1..l_r: normalisers
        n_rej, n_expl = dsp.dspark_verify_residual_rows(head.dims, rnd.ws_verify)
        vbytes += n_rej * row                           # rejected row: rescanned for its trials
        vbytes += n_expl * (2 * row + r * 2)            # explicit residual: target + base, E row
        vbytes += (V * r * 2) if n_expl else 0          # W2t once for the explicit pass
        vbytes += int((~rejected).sum()) * row          # bonus row of the rest
        # (each trial's 256 target ids, W2t row and base logit, ~1.5 KB, not counted)
    else:
        n_rej = n_expl = 0
        vbytes = int((ln + 1).sum()) * row             # rows 1..l_r + 1: argmaxes
    verify_gbs = vbytes / (stage["verify"] * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": job_throughput(R * G, ms, ws), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "R": R, "gamma": G, "V": V, "r": r, "d": d, "tau": w.tau,
                   "l2": "inputs larger than L2 (LM head 1.85 GB streamed every step)"
                   if V * d * 2 > 129e6 else "L2 not flushed",
                   "parallelism": f"replicas x{ws}"},
        "rounds_per_s": ws / (ms * 1e-3),
        "stages_ms": stage,
        "admitted_K": K_adm, "mean_accepted": acc,
        "roofline": lm_roof,
        "markov_loop_roofline": markov_roof,
        "markov_loop_hbm": {"achieved": markov_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": markov_gbs / peaks["hbm_gbs"]},
        "verify_hbm": {"bytes": vbytes, "achieved": verify_gbs, "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": verify_gbs / peaks["hbm_gbs"],
                       **({"rejected_rows": n_rej, "explicit_rows": n_expl} if w.tau > 0
                          else {})},
        "gpu_launches": launches,
        "clocks": clk,
    }

    if args.fused_variant:
        # the fused single-contraction draft step in place of LM head + Markov loop:
        # per step one GEMM [R, d + r] x [d + r, V] (W_lm and W2t streamed each step)
        W_cat = torch.empty((V, d + r), dtype=torch.bfloat16, device="cuda")
        dsp.dspark_pack_fused(dims, head.W_lm, head.W2t, W_cat)
        fws = dsp.workspace(dsp.dspark_fused_workspace_bytes(dims))

        def fused():
            dsp.dspark_fused_draft(dims, h, anchor, W_cat, head.W1, head.w_conf, head.T, tau, ds,
                                   rnd.tokens, rnd.conf, rnd.logp_d, rnd.lse_d, fws)

        for _ in range(3):
            fused()
        torch.cuda.synchronize()
        n_f = max(3, min(args.steps, 50))
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("fused")
        f0.record(stream)
        for _ in range(n_f):
            fused()
        f1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        dsp.check_device_status()
        fms = f0.elapsed_time(f1) / n_f
        fbytes = G * (V * (d + r) * 2 + R * (d + r) * 2)
        line["fused_variant"] = {
            "draft_ms": fms, "lm_head_plus_loop_ms": stage["lm_head"] + stage["markov_loop"],
            "draft_bytes": fbytes, "hbm_frac": fbytes / (fms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "tensor_frac": G * 2.0 * R * (d + r) * V / (fms * 1e-3) / 1e12 / tc_peak}
        del W_cat, fws

    if args.rnn_variant:
        # the RNN head in place of the Markov head (untrained weights of the
        # stated shapes: W_rec [2r, 2r], W_hid [2r, d], std 1/sqrt(fan-in))
        g = torch.Generator(device="cuda").manual_seed(w.seed + 17)
        W_rec = (torch.randn((2 * r, 2 * r), generator=g, device="cuda") /
                 math.sqrt(2 * r)).to(torch.bfloat16)
        W_hid = (torch.randn((2 * r, d), generator=g, device="cuda") /
                 math.sqrt(d)).to(torch.bfloat16)
        rws = dsp.workspace(dsp.dspark_rnn_workspace_bytes(dims))

        def rnn():
            dsp.dspark_rnn_draft(dims, rnd.base, h, anchor, head.W1, head.W2t, W_rec, W_hid,
                                 head.w_conf, head.T, tau, ds, rnd.tokens, rnd.conf, rnd.logp_d,
                                 rnd.lse_d, rws)

        for _ in range(3):
            rnn()
        torch.cuda.synchronize()
        n_r = max(3, min(args.steps, 50))
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("rnn")
        r0.record(stream)
        for _ in range(n_r):
            rnn()
        r1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        dsp.check_device_status()
        line["rnn_variant"] = {"draft_ms": r0.elapsed_time(r1) / n_r,
                               "markov_loop_ms": stage["markov_loop"]}
        del W_rec, W_hid, rws

    if args.sts_fit:
        # one Sequential Temperature Scaling fit: 1M held-out rounds, gamma
        # positions, 51 temperatures, 15 bins (synthetic logits and acceptances)
        N = 1 << 20
        g = torch.Generator(device="cuda").manual_seed(w.seed + 29)
        z = (1.2 + 2.0 * torch.randn((N, G), generator=g, device="cuda")).contiguous()
        accepted = torch.randint(0, G + 1, (N,), generator=g, device="cuda", dtype=torch.int32)
        grid = torch.linspace(0.5, 3.0, 51, device="cuda")
        T_out = torch.empty(G, dtype=torch.float32, device="cuda")
        ece = torch.empty(G, dtype=torch.float64, device="cuda")
        sws = dsp.workspace(dsp.dspark_sts_workspace_bytes(N, G, 51, 15))
        for _ in range(3):
            dsp.dspark_sts_fit(z, accepted, grid, 15, T_out, ece, sws)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.nvtx.range_push("sts")
        s0.record(stream)
        for _ in range(10):
            dsp.dspark_sts_fit(z, accepted, grid, 15, T_out, ece, sws)
        s1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        dsp.check_device_status()
        line["sts_fit"] = {"ms": s0.elapsed_time(s1) / 10, "rounds": N, "grid": 51, "bins": 15}
        del z, accepted, sws

    if not args.no_e2e:
        # end to end through the public API from pinned host buffers
        h_host = h.cpu().pin_memory()
        a_host = anchor.cpu().pin_memory()
        t_host = target.cpu().pin_memory()
        dev_in = {"h": torch.empty_like(h), "anchor": torch.empty_like(anchor),
                  "target": torch.empty_like(target)}
        out_host = {k: torch.empty(getattr(rnd, k).shape, dtype=getattr(rnd, k).dtype,
                                   pin_memory=True)
                    for k in ("tokens", "len", "accepted", "bonus")}
        for _ in range(2):
            rnd.run_host(h_host, a_host, t_host, sps, tau, ds, vs, dev_in, out_host)
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            rnd.run_host(h_host, a_host, t_host, sps, tau, ds, vs, dev_in, out_host)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
        bi = h.numel() * 2 + anchor.numel() * 4 + target.numel() * 2
        bo = sum(t.numel() * t.element_size() for t in out_host.values())
        line["e2e"] = {"value": job_throughput(R * G, ems, ws), "unit": UNIT,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_sample)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_setup()
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py: the DSpark CUDA path needs a GPU")
        run_dspark(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
