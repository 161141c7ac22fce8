#!/usr/bin/env python3
"""Benchmark: chunkwise delta-rule forward tokens/s (+ roofline) and decode-step GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Workload (default ``gdn_kla_bf16``): B=8, H=8, T=2048, dk=dv=128, chunk 64,
bf16 q/k/v, fp32 gates and state, GDN and KLA on the same seeded inputs.  One
step is one chunkwise forward over the whole batch for each of the two
variants (each a prep and a carry launch of libdr); ``value`` counts B*T tokens
per variant pass.  ``--workload`` times any other workload of
``recurrent_associative_memory_gb300.workloads`` (PGDN, the per-channel-decay
variants, the exact Kalman memory, the 64K-token prefill) the same way.  Inputs are resident in HBM before the timed region; L2 is
flushed (a 256 MiB write) between timed steps and the flush is not timed.

The same JSON line carries:
  roofline      the forward kernel's algorithmic bytes / CUDA-event time vs the
                measured HBM peak in MEASURED_PEAKS.json;
  decode        dr_decode_step at batch 256, H=16, d=128 (KLA): HBM GB/s of the
                algorithmic bytes (state read + write, q/k/v/o, gates);
  e2e           the same forward metric with pinned host buffers: every step
                copies its inputs H2D, runs both forwards and copies both
                outputs D2H, all inside the timed region; the copies run on
                their own streams into double-buffered device tensors, so step
                i+1's inputs arrive and step i-1's outputs leave while step i
                computes;
  cpu_baseline  the fp64 oracle (numpy, tokenwise) on a bounded sample of the
                workload (one batch row, all heads), on the host cores;
  clocks        nvidia-smi SM clocks and throttle reasons sampled during the
                timed region.

N > 1 (torchrun): every rank runs its own full replica of the workload (no
data-path collective; weak scaling); the step time is the max over ranks and
``value`` sums the ranks' tokens.  ``--impl reference`` times the fp64 oracle
on the host cores instead (rank 0 only) and prints the same kind of line.
"""

from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunkwise delta-rule fwd tokens/s & % roofline; decode-step HBM GB/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gdn_kla_bf16")
    p.add_argument("--decode-steps", type=int, default=200)
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-heads", type=int, default=8)
    return p.parse_args()


KERNEL_SOURCES = {
    "chunk_tc_split": ["chunk_tc_split.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_tc_ws": ["chunk_tc_ws.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_tc": ["chunk_tc.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_simt": ["chunk_simt.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh", "chain.cuh"],
    "decode": ["decode.cu", "dr_common.cuh"],
    "kalman": ["kalman.cu", "dr_common.cuh"],
}


def source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "recurrent_associative_memory_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel, workload, variant=None):
    """DRAM bytes per launch from the ncu capture recorded in profiles/traffic.json,
    or None when there is none or the kernel source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("source_sha256") != source_hash(kernel):
        return None
    variants = rec.get("variants", [rec.get("variant")])
    if rec.get("workload") != workload or (variant and variant not in variants):
        return None
    return rec.get("dram_bytes_per_launch")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


# ---------------------------------------------------------------- algorithmic bytes

def fwd_bytes(wl, variant, with_final=True):
    """Bytes a forward launch must move: q,k,v in, o out, gates, final state (+aux)."""
    el = 2 if wl.dtype == "bf16" else 4
    ht = wl.B * wl.T * wl.H
    per_ht = (2 * wl.dk + 2 * wl.dv) * el          # q, k, v, o
    gates = {"gdn": 8, "kla": 8, "pgdn": 16, "kdn": 8 * wl.dk + 4,
             "kda": 4 * wl.dk + 4, "pkda": 4 * wl.dk + 12, "ikdn": 4 * wl.dk + 8,
             "ekdn": 8 * wl.dk + 4}[variant]
    total = ht * (per_ht + gates)
    if variant in ("pgdn", "pkda"):
        total += wl.H * 4
    if with_final:
        total += wl.B * wl.H * wl.dk * wl.dv * 4
        if variant in ("pgdn", "kdn", "pkda"):
            total += wl.B * wl.H * wl.dk * 4
        if variant == "ikdn":   # one variance per head
            total += wl.B * wl.H * 4
        if variant == "ekdn":   # the dense covariance
            total += wl.B * wl.H * wl.dk * wl.dk * 4
    return total


def decode_bytes(wl):
    el = 2 if wl.dtype == "bf16" else 4
    bh = wl.B * wl.H
    return bh * (2 * wl.dk * wl.dv * 4 + (2 * wl.dk + 2 * wl.dv) * el + 8)


def kernels_per_call(path, variant, B, H, has_workspace, nsm):
    """libdr kernels one dr_chunk_fwd call launches on ``path``.

    The two-phase paths launch a prep and a carry kernel; PGDN adds its key
    statistic's map and scan kernels; on the CUDA-core two-phase path a few
    rows (3 B H < nsm) make Diagonal KDN add its variance map and scan kernels
    and PKDA / isotropic KDN run the fused kernel alone (KDA: never either).
    Every other path is one kernel.  A memset of the chain flags is not a kernel.
    """
    if not has_workspace or path not in ("tc_split", "simt_split"):
        return 1
    if path == "simt_split":
        if 3 * B * H >= nsm or variant == "kda":
            return 2
        return 1 if variant in ("pkda", "ikdn") else 4
    return 4 if variant == "pgdn" else 2


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to a temporary file, or where DR_BENCH_CLOCKS_DIR says
        out_dir = os.environ.get("DR_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU baseline)

def _oracle_heads(args):
    name, variant, heads = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np  # noqa: F401
    import oracle
    from recurrent_associative_memory_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    inp = W.generate(W.small(name, B=1), variant)      # batch row 0 of the same distributions
    f = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    sl = lambda t: None if t is None else f(t[:, :, heads])  # noqa: E731
    t0 = time.perf_counter()
    oracle.tokenwise(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["log_alpha"]), variant,
                     eta=sl(inp.get("eta")), eps=wl.eps, q_l2norm=wl.q_l2norm,
                     k_l2norm=wl.k_l2norm, alphaP=sl(inp.get("alphaP")),
                     betaP=sl(inp.get("betaP")),
                     mu=None if inp.get("mu") is None else f(inp["mu"][heads]),
                     omega=sl(inp.get("omega")), r=sl(inp.get("r")), info_scale=wl.info_scale)
    return time.perf_counter() - t0


def oracle_sample(name, n_heads, pool=None):
    """Time the oracle on one batch row (n_heads heads) for every variant of the workload.

    Returns (tokens, seconds, cores): tokens counted like the GPU metric
    (B*T per variant pass, scaled by the fraction of heads sampled)."""
    from recurrent_associative_memory_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    n_heads = min(n_heads, wl.H)
    jobs = [(name, v, [h]) for v in wl.variants for h in range(n_heads)]
    t0 = time.perf_counter()
    if pool is not None:
        list(pool.map(_oracle_heads, jobs))
        cores = min(pool._processes, len(jobs))
    else:
        for j in jobs:
            _oracle_heads(j)
        cores = 1
    secs = time.perf_counter() - t0
    tokens = len(wl.variants) * wl.T * n_heads / wl.H
    return tokens, secs, cores


# ---------------------------------------------------------------- distributed helpers

# One process per GPU; the ranks run independent replicas (the forward shards over
# (b, h) with no exchange), so the only collectives are the timing barrier and the
# max of the ranks' times.  NCCL on GPUs; gloo when no GPU is present (CPU tests).

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, steps, n_variants, B, T, seconds):
    """Whole-job throughput: every rank runs the same workload, so the job moves
    world x steps x variants x B x T tokens in the slowest rank's time."""
    return world * steps * n_variants * B * T / seconds


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from recurrent_associative_memory_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    ctx = mp.get_context("spawn")
    ncores = os.cpu_count() or 1
    n_heads = min(args.cpu_sample_heads, wl.H)
    with ctx.Pool(min(ncores, n_heads * len(wl.variants))) as pool:
        for _ in range(args.warmup):
            oracle_sample(args.workload, n_heads, pool)
        tok, secs, cores = 0.0, 0.0, 1
        for _ in range(args.steps):
            t_, s_, cores = oracle_sample(args.workload, n_heads, pool)
            tok += t_
            secs += s_
    value = tok / secs
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.dk,
                       "dv": wl.dv, "chunk": wl.chunk, "variants": list(wl.variants)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"fp64 tokenwise oracle, batch row 0, {n_heads} of {wl.H} "
                                       f"heads, T={wl.T}, variants {list(wl.variants)}, per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm

def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    # the oracle pool must exist before the first CUDA call (spawn context anyway)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = mp.get_context("spawn").Pool(min(os.cpu_count() or 1, 16))

    import torch
    from recurrent_associative_memory_gb300 import dr, runner
    from recurrent_associative_memory_gb300 import workloads as W

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pk = peaks()
    wl = W.WORKLOADS[args.workload]
    variants = list(wl.variants)

    # inputs: shared q/k/v, per-variant gates, generated on the CPU then copied
    host = {v: W.generate(wl, v) for v in variants}
    dev = {v: runner.to_device(host[v]) for v in variants}
    outs = {v: torch.empty(wl.B, wl.T, wl.H, wl.dv, dtype=dev[v]["q"].dtype, device="cuda")
            for v in variants}
    finals = {v: torch.empty(wl.B, wl.H, wl.dk, wl.dv, dtype=torch.float32, device="cuda")
              for v in variants}
    auxf = {v: (torch.empty(wl.B, wl.H, wl.dk, device="cuda") if v in ("pgdn", "kdn") else None)
            for v in variants}
    # one caller-owned workspace, reused by the variants' calls in stream order
    wss = [runner.workspace_for(dev[v]) for v in variants]
    ws = max((w for w in wss if w is not None), key=lambda w: w.numel(), default=None)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        for v in variants:
            runner.chunk_fwd(dev[v], out=outs[v], final_state=finals[v], aux_final=auxf[v],
                             stream=stream, workspace=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    dr.check(dr.dr_get_device_status(), "warmup")

    # timed region: per-step events around the forwards; L2 flush between steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    vev = {v: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for v in variants}
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        for v in variants:
            vev[v][i][0].record(stream)
            runner.chunk_fwd(dev[v], out=outs[v], final_state=finals[v], aux_final=auxf[v],
                             stream=stream, workspace=ws)
            vev[v][i][1].record(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in ev]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    dr.check(dr.dr_get_device_status(), "timed region")
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    launches = args.steps * sum(
        kernels_per_call(dr.dr_chunk_fwd_path(dr.VARIANT_IDS[v], 1 if wl.dtype == "bf16" else 0,
                                              wl.dk, wl.dv, wl.chunk),
                         v, wl.B, wl.H, ws is not None, nsm)
        for v in variants)
    value = job_tokens_per_s(world, args.steps, len(variants), wl.B, wl.T, total_s)

    var_stats = {}
    for v in variants:
        ms = statistics.mean(s.elapsed_time(e) for s, e in vev[v])
        byt = fwd_bytes(wl, v)
        var_stats[v] = {"ms": ms, "tokens_per_s": wl.B * wl.T / (ms / 1e3),
                        "gbs": byt / (ms / 1e3) / 1e9,
                        "frac_hbm": byt / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                        "path": dr.dr_chunk_fwd_path(dr.VARIANT_IDS[v], 1 if wl.dtype == "bf16"
                                                     else 0, wl.dk, wl.dv, wl.chunk)}
    dom = max(variants, key=lambda v: var_stats[v]["ms"])
    byt = fwd_bytes(wl, dom)
    ach = byt / (var_stats[dom]["ms"] / 1e3) / 1e9
    kname = "chunk_" + var_stats[dom]["path"]
    kdesc = f"{kname} ({dom})"
    if var_stats[dom]["path"] == "tc_split":
        kdesc = f"{kname}: chunk_prep + chunk_carry of one dr_chunk_fwd call ({dom})"
    roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "traffic": measured_traffic(kname, wl.name, dom),
            "kernel": kdesc,
            "algorithmic_bytes_per_launch": byt, "peak_source": pk["src"]}

    result = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
              "steps": args.steps, "warmup": max(3, args.warmup),
              "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
              "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.dk,
                         "dv": wl.dv, "chunk": wl.chunk, "variants": variants,
                         "state": "fp32", "l2": "flushed between timed steps (256 MiB write)",
                         "parallelism": f"replicas x{world}"},
              "roofline": roof, "variants": var_stats, "gpu_launches": launches, "clocks": clk}

    # ---- decode step (batch 256, H 16): HBM GB/s
    if not args.no_decode:
        dwl = W.WORKLOADS["kla_decode_bf16"]
        pool_steps = [runner.to_device(W.generate_decode_step(dwl, s)) for s in range(8)]
        S = torch.zeros(dwl.B, dwl.H, dwl.dk, dwl.dv, device="cuda")
        S.normal_(0, 0.05)
        dout = torch.empty(dwl.B, dwl.H, dwl.dv, dtype=torch.bfloat16, device="cuda")
        for i in range(5):
            runner.decode_step(pool_steps[i % 8], S, out=dout, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.decode_steps):
            runner.decode_step(pool_steps[i % 8], S, out=dout, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        dr.check(dr.dr_get_device_status(), "decode")
        ms = e0.elapsed_time(e1) / args.decode_steps
        db = decode_bytes(dwl)
        gbs = db / (ms / 1e3) / 1e9
        result["decode"] = {"workload": dwl.name, "B": dwl.B, "H": dwl.H, "d": dwl.dk,
                            "ms_per_step": ms, "gbs": gbs, "frac": gbs / pk["hbm_gbs"],
                            "algorithmic_bytes_per_step": db, "steps": args.decode_steps,
                            "traffic": measured_traffic("decode", dwl.name),
                            "tokens_per_s": dwl.B / (ms / 1e3), "launches": args.decode_steps}

    # ---- end to end through the public API with pinned host buffers
    if not args.no_e2e:
        keys = [k for k in dev[variants[0]] if torch.is_tensor(dev[variants[0]][k])]
        hpin = {v: {k: host[v][k].pin_memory() for k in keys} for v in variants}
        hout = {v: torch.empty_like(outs[v], device="cpu").pin_memory() for v in variants}
        h2d = sum(hpin[variants[0]][k].numel() * hpin[variants[0]][k].element_size()
                  for k in ("q", "k", "v"))
        h2d += sum(hpin[v][k].numel() * hpin[v][k].element_size()
                   for v in variants for k in keys if k not in ("q", "k", "v"))
        d2h = sum(hout[v].numel() * hout[v].element_size() for v in variants)

        # two device buffer sets: set i & 1 takes step i's inputs and outputs
        sets = [dev, {v: {k: (t.clone() if torch.is_tensor(t) else t) for k, t in dev[v].items()}
                      for v in variants}]
        osets = [outs, {v: torch.empty_like(outs[v]) for v in variants}]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("h2d", "fwd", "d2h")}

        def e2e_step(i):
            s_ = i & 1
            d_in = sets[s_]
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev["fwd"][s_])     # step i-2 has read set s_
                for k in ("q", "k", "v"):
                    d_in[variants[0]][k].copy_(hpin[variants[0]][k], non_blocking=True)
                for v in variants:
                    for k in keys:
                        if k not in ("q", "k", "v"):
                            d_in[v][k].copy_(hpin[v][k], non_blocking=True)
                ev["h2d"][s_].record(h2d_s)
            stream.wait_event(ev["h2d"][s_])
            if i >= 2:
                stream.wait_event(ev["d2h"][s_])        # step i-2's outputs have left set s_
            for v in variants:
                d = dict(d_in[v])
                for k in ("q", "k", "v"):
                    d[k] = d_in[variants[0]][k]
                runner.chunk_fwd(d, out=osets[s_][v], final_state=finals[v], aux_final=auxf[v],
                                 stream=stream, workspace=ws)
            ev["fwd"][s_].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev["fwd"][s_])
                for v in variants:
                    hout[v].copy_(osets[s_][v], non_blocking=True)
                ev["d2h"][s_].record(d2h_s)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(5, min(args.steps, 20))
        e0.record(h2d_s)
        for i in range(n):
            e2e_step(i)
        e1.record(d2h_s)                                # after the last step's D2H
        torch.cuda.synchronize()
        sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
        result["e2e"] = {"value": world * n * len(variants) * wl.B * wl.T / sec, "unit": "tokens/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}

    if pool is not None:
        n_heads = min(args.cpu_sample_heads, wl.H)
        tok, secs, cores = oracle_sample(args.workload, n_heads, pool)
        pool.close()
        result["cpu_baseline"] = {"value": tok / secs, "unit": "tokens/s", "cores": cores,
                                  "kind": "oracle",
                                  "sample": f"fp64 tokenwise oracle on batch row 0, {n_heads} of "
                                            f"{wl.H} heads, T={wl.T}, variants {variants}"}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
