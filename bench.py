#!/usr/bin/env python3
"""Benchmark: chunkwise delta-rule forward tokens/s (+ roofline) and decode-step GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-configs] [--no-decode] [--no-e2e]
                    [--no-cpu-baseline]

Headline workload (default ``gdn_kla_bf16``): B=8, H=8, T=2048, dk=dv=128,
chunk 64, bf16 q/k/v, fp32 gates and state, GDN and KLA on the same seeded
inputs.  One step is one chunkwise forward over the whole batch for each of the
two variants (each a prep and a carry launch of libdr); ``value`` counts B*T
tokens per variant pass.  ``--workload`` makes any other workload of
``recurrent_associative_memory_gb300.workloads`` the headline.  Inputs are
resident in HBM before the timed region; L2 is flushed (a 256 MiB write)
between timed steps and the flush is not timed.

The same JSON line carries:
  roofline      the forward's algorithmic bytes / CUDA-event time vs the
                measured HBM peak in MEASURED_PEAKS.json;
  configs       every workload the method's configurations name, each timed the
                same way (CUDA events, L2 flushed between steps): the fp32
                parity case, GDN and KLA, PGDN, Diagonal KDN, the 64K-token KLA
                prefill and the batch-256 decode step; per entry the time,
                tokens/s, algorithmic bytes, roofline fraction, the recorded DRAM
                traffic where an ncu capture exists, and the largest
                max|gpu - oracle| / max|oracle| over sampled (b, h) rows of the
                output, the final state and the gain state;
  decode        dr_decode_step at batch 256, H=16, d=128 (KLA), and per variant
                (GDN, PGDN, Diagonal KDN, KDA, PKDA, isotropic KDN, exact Kalman):
                HBM GB/s of the algorithmic bytes (state read + write, q/k/v/o,
                gates, gain state);
  e2e           the headline metric with pinned host buffers: every step copies
                its inputs H2D, runs both forwards and copies both outputs D2H,
                all inside the timed region; the copies run on their own streams
                into double-buffered device tensors, so step i+1's inputs arrive
                and step i-1's outputs leave while step i computes;
  cpu_baseline  the fp64 oracle (numpy, tokenwise) on a bounded sample of the
                headline workload (batch row 0, all heads, both variants,
                repeated), on the host cores, in a spawn pool warmed first (the
                inputs are drawn once per worker, outside the timed calls); also
                the same oracle on one core;
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

# The workloads of the method's configurations, in their order: the fp32 parity
# case, GDN vs KLA, PGDN, Diagonal KDN, the long-context prefill, then decode.
CONFIG_WORKLOADS = [("0", "kla_fp32_small"), ("1", "gdn_kla_bf16"), ("2", "pgdn_bf16"),
                    ("3", "kdn_bf16"), ("4a", "kla_prefill_bf16"), ("4b", "kla_decode_bf16")]
# the per-channel-decay and exact-Kalman rows beyond the configurations: forward
# (and, where it exists, backward) timed on their own workloads with oracle parity
NEXT_WORKLOADS = [("kda", "kda_bf16"), ("pkda", "pkda_bf16"), ("ikdn", "ikdn_bf16"),
                  ("ekdn", "ekdn_bf16")]
BWD_VARIANTS = ("gdn", "kla", "pgdn", "kda", "kdn", "pkda", "ikdn")
# decode-step variants timed besides the headline KLA step, on their own workloads' flags
DECODE_VARIANTS = {"gdn": "gdn_kla_bf16", "pgdn": "pgdn_bf16", "kdn": "kdn_bf16",
                   "kda": "kda_bf16", "pkda": "pkda_bf16", "ikdn": "ikdn_bf16",
                   "ekdn": "ekdn_bf16"}


def parse(argv=None):
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
    p.add_argument("--no-configs", action="store_true")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-next", action="store_true",
                   help="skip the KDA / PKDA / isotropic KDN / exact Kalman rows")
    p.add_argument("--cpu-sample-heads", type=int, default=8)
    p.add_argument("--cpu-sample-reps", type=int, default=10)
    return p.parse_args(argv)


KERNEL_SOURCES = {
    "chunk_tc_split": ["chunk_tc_split.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_tc_ws": ["chunk_tc_ws.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_tc": ["chunk_tc.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh"],
    "chunk_simt": ["chunk_simt.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh", "chain.cuh"],
    "chunk_simt_split": ["chunk_simt.cu", "umma.cuh", "tc_common.cuh", "dr_common.cuh", "chain.cuh"],
    "chunk_tc_pc_split": ["chunk_tc_pc.cu", "chunk_simt.cu", "chunk_tc_split.cu", "umma.cuh",
                          "tc_common.cuh", "dr_common.cuh", "chain.cuh"],
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
    if not rec or kernel not in KERNEL_SOURCES or rec.get("source_sha256") != source_hash(kernel):
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

def gate_bytes(variant, dk):
    """fp32 gate bytes per (b, t, h): what the variant's write rule reads."""
    return {"gdn": 8, "kla": 8, "pgdn": 16, "kdn": 8 * dk + 4, "kda": 4 * dk + 4,
            "pkda": 4 * dk + 12, "ikdn": 4 * dk + 8, "ekdn": 8 * dk + 4}[variant]


def aux_elems(variant, dk):
    """fp32 elements of the gain state per (b, h) (0: none)."""
    return {"pgdn": dk, "kdn": dk, "pkda": dk, "ikdn": 1, "ekdn": dk * dk}.get(variant, 0)


def aux_shape(variant, B, H, dk):
    n = aux_elems(variant, dk)
    if n == 0:
        return None
    return {1: (B, H), dk: (B, H, dk), dk * dk: (B, H, dk, dk)}[n]


def fwd_bytes(wl, variant, with_final=True):
    """Bytes a forward launch must move: q,k,v in, o out, gates, final state (+aux)."""
    el = 2 if wl.dtype == "bf16" else 4
    ht = wl.B * wl.T * wl.H
    per_ht = (2 * wl.dk + 2 * wl.dv) * el          # q, k, v, o
    total = ht * (per_ht + gate_bytes(variant, wl.dk))
    if variant in ("pgdn", "pkda"):
        total += wl.H * 4
    if with_final:
        total += wl.B * wl.H * (wl.dk * wl.dv + aux_elems(variant, wl.dk)) * 4
    return total


def bwd_bytes(wl, variant="kla"):
    """Bytes one backward call must move: q, k, v and dL/do in (the input dtype) and
    the gates; dq, dk, dv (fp32) and the gates' gradients out (the same sizes as
    the gates: per-channel decay gives d log alpha per channel); the initial state
    and dL/dS_T in, dL/dS_0 out; the gain state's initial value and dL/d(final) in
    and its gradient out (PGDN / PKDA: also mu in and dL/dmu out)."""
    el = 2 if wl.dtype == "bf16" else 4
    ht = wl.B * wl.T * wl.H
    gates = gate_bytes(variant, wl.dk)
    per_ht = (2 * wl.dk + 2 * wl.dv) * el + gates + (2 * wl.dk + wl.dv) * 4 + gates
    total = ht * per_ht + 3 * wl.B * wl.H * wl.dk * wl.dv * 4
    total += 3 * wl.B * wl.H * aux_elems(variant, wl.dk) * 4
    if variant in ("pgdn", "pkda"):
        total += 2 * wl.H * 4
    return total


def bwd_kernels_per_call(variant, B=1, H=1, nsm=152):
    """libdr kernels one dr_chunk_bwd call launches: the forward again (prep and
    carry; PGDN also its statistic's map and scan; Diagonal KDN with few rows,
    3 B H < SMs, its variance map and scan), the reverse carry, the state
    products, the local gradients, then the gain's adjoint (each chunk's affine
    map, the scan over chunks, each chunk's gradients; PGDN / PKDA also the d mu
    sum)."""
    fwd = {"pgdn": 4, "kdn": 2 if 3 * B * H >= nsm else 4}.get(variant, 2)
    gain = {"pgdn": 4, "pkda": 4, "kdn": 3, "ikdn": 3}.get(variant, 0)
    return fwd + 3 + gain


def decode_bytes(wl, variant="kla"):
    """Bytes one decode step must move: the state (and gain state) read and written
    once, q, k, v in and o out, the step's gates."""
    el = 2 if wl.dtype == "bf16" else 4
    bh = wl.B * wl.H
    per_bh = (2 * (wl.dk * wl.dv + aux_elems(variant, wl.dk)) * 4 + (2 * wl.dk + 2 * wl.dv) * el
              + gate_bytes(variant, wl.dk))
    return bh * per_bh + (wl.H * 4 if variant in ("pgdn", "pkda") else 0)


def kernels_per_call(path, variant, B, H, has_workspace, nsm, NC=0):
    """libdr kernels one dr_chunk_fwd call launches on ``path``.

    The two-phase paths launch a prep and a carry kernel; PGDN adds its key
    statistic's map and scan kernels; on the CUDA-core two-phase path a few
    rows (3 B H < nsm) make Diagonal KDN add its variance map and scan kernels
    and PKDA / isotropic KDN run the fused kernel alone (KDA: never either).
    Every other path is one kernel.  A memset of the chain flags is not a kernel.
    """
    if not has_workspace or path not in ("tc_split", "simt_split", "tc_pc_split"):
        return 1
    if path in ("simt_split", "tc_pc_split"):
        if 3 * B * H >= nsm or variant == "kda":
            return 2
        return 1 if variant in ("pkda", "ikdn") else 4
    n = 4 if variant == "pgdn" else 2
    return n + 2 if seg_segments(nsm, B * H, NC) else n


def seg_segments(nsm, rows, NC):
    """Segments per row of the tensor-core path's segment-parallel carry (0: not
    used).  With few rows (6 rows <= SMs) the carry runs as a first pass, a
    composition of segment start states and a replay pass (two more launches);
    the library picks the largest G <= (SMs / rows - 2) / 4 + 2 (at most 64,
    at least 3) whose segments of ceil(NC / G) chunks are >= 2 long and all
    non-empty."""
    if nsm <= 0 or rows * 6 > nsm:
        return 0
    G = min((nsm // rows - 2) // 4 + 2, 64)
    for g in range(G, 2, -1):
        Ls = -(-NC // g)
        if Ls >= 2 and (g - 1) * Ls < NC:
            return g
    return 0


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


# ---------------------------------------------------------------- oracle (pool workers)
# These run in spawned worker processes (never in the process that drives the GPU).

_INPUT_CACHE = {}


def _oracle_call(inp, variant, S0=None, aux0=None):
    """The fp64 tokenwise oracle on one input dict of numpy arrays."""
    import numpy as np
    import oracle
    f = lambda t: None if t is None else np.asarray(t, dtype=np.float64)  # noqa: E731
    return oracle.tokenwise(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_alpha"]), variant,
                            eta=f(inp.get("eta")), eps=inp["eps"], q_l2norm=inp["q_l2norm"],
                            k_l2norm=inp["k_l2norm"], alphaP=f(inp.get("alphaP")),
                            betaP=f(inp.get("betaP")), mu=f(inp.get("mu")), x=inp["x"],
                            log_floor=inp["log_floor"], omega=f(inp.get("omega")),
                            r=f(inp.get("r")), info_scale=inp["info_scale"], S0=f(S0),
                            aux0=f(aux0))


def _sample_inputs(name, variant, head):
    """Batch row 0, one head of a workload's inputs (drawn once per worker)."""
    key = (name, variant)
    if key not in _INPUT_CACHE:
        from recurrent_associative_memory_gb300 import workloads as W
        full = W.generate(W.small(name, B=1), variant)
        _INPUT_CACHE[key] = full
    full = _INPUT_CACHE[key]
    return {k: (t[:, :, head:head + 1].float().numpy() if k != "mu" else
                t[head:head + 1].float().numpy()) if hasattr(t, "numpy") else t
            for k, t in full.items()}


def _oracle_timed(job):
    """Worker: run the oracle on one sampled head; return the seconds of the call only."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    name, variant, head = job
    inp = _sample_inputs(name, variant, head)
    t0 = time.perf_counter()
    _oracle_call(inp, variant)
    return time.perf_counter() - t0


def _oracle_bwd_parity(job):
    """Worker: the oracle's reverse sweep (every gradient) for one sliced row."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np
    from oracle import backward as obw
    tag, inp, variant, dO, dS, S0 = job
    f = lambda t: None if t is None else np.asarray(t, dtype=np.float64)  # noqa: E731
    g = obw.tokenwise_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_alpha"]),
                               variant, f(dO), f(dS), eta=f(inp.get("eta")), eps=inp["eps"],
                               q_l2norm=inp["q_l2norm"], k_l2norm=inp["k_l2norm"], S0=f(S0),
                               alphaP=f(inp.get("alphaP")), betaP=f(inp.get("betaP")),
                               mu=f(inp.get("mu")), x=inp.get("x", 1.5),
                               log_floor=inp.get("log_floor", 1e-12), omega=f(inp.get("omega")),
                               r=f(inp.get("r")), info_scale=inp.get("info_scale", 1.0))
    if variant in ("kdn", "ikdn"):
        names = ("dq", "dk", "dv", "dlog_alpha", "dS0", "domega", "dr")
    else:
        names = ("dq", "dk", "dv", "dlog_alpha", "deta", "dS0")
        if variant in ("pgdn", "pkda"):
            names += ("dalphaP", "dbetaP")
    return tag, {k: g[k] for k in names}


def _oracle_parity(job):
    """Worker: the oracle's output, final state and gain state for one sliced row."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    tag, inp, variant, S0, aux0 = job
    o, S, aux = _oracle_call(inp, variant, S0, aux0)
    return tag, o, S, aux


def oracle_sample(name, n_heads, pool, reps=1):
    """Time the oracle on batch row 0 (n_heads heads, every variant of the workload).

    The workers draw the inputs on their first call, so the caller warms the pool
    with one call first; afterwards only the oracle runs inside the timed wall.
    Returns (tokens, wall seconds, worker seconds, cores): tokens counted like the
    GPU metric (B*T per variant pass, scaled by the fraction of heads sampled)."""
    from recurrent_associative_memory_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    n_heads = min(n_heads, wl.H)
    jobs = [(name, v, h) for _ in range(reps) for v in wl.variants for h in range(n_heads)]
    t0 = time.perf_counter()
    per_job = list(pool.map(_oracle_timed, jobs, chunksize=1))
    secs = time.perf_counter() - t0
    cores = min(pool._processes, len(jobs))
    tokens = reps * len(wl.variants) * wl.T * n_heads / wl.H
    return tokens, secs, sum(per_job), cores


def oracle_one_core(name, pool):
    """The oracle on one core: every variant of one head, one job after another in a
    single worker.  Returns tokens/s in the metric's units."""
    from recurrent_associative_memory_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    secs = sum(pool.apply(_oracle_timed, ((name, v, 0),)) for v in wl.variants)
    return len(wl.variants) * wl.T / wl.H / secs


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

def cpu_sample_text(wl, n_heads, reps):
    return (f"fp64 tokenwise oracle, batch row 0, {n_heads} of {wl.H} heads, T={wl.T}, "
            f"variants {list(wl.variants)}, x{reps}, warmed spawn pool (inputs drawn once "
            f"per worker, outside the timed calls)")


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
            t_, s_, _, cores = oracle_sample(args.workload, n_heads, pool)
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
                             "sample": cpu_sample_text(wl, n_heads, 1) + ", per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm: helpers

def rel_err(x, ref):
    import numpy as np
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = float(np.abs(ref).max())
    return float(np.abs(x - ref).max() / d) if d > 0 else float(np.abs(x).max())


def sampled_pairs(B, H, n):
    out = []
    for p in [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]:
        if p not in out:
            out.append(p)
    return out[:n]


def slice_row(inp, b, h):
    """One (b, h) row of a CPU input dict as [1, T, 1, d] numpy arrays (+ flags)."""
    out = {}
    for k, t in inp.items():
        if not hasattr(t, "numpy"):
            out[k] = t
        elif k == "mu":
            out[k] = t[h:h + 1].float().numpy()
        else:
            out[k] = t[b:b + 1, :, h:h + 1].float().numpy()
    return out


class Forward:
    """One workload's device inputs, outputs and workspace, and its timed forward."""

    def __init__(self, torch, dr, runner, W, wl, host=None):
        self.torch, self.dr, self.runner, self.wl = torch, dr, runner, wl
        self.variants = list(wl.variants)
        self.host = host or {v: W.generate(wl, v) for v in self.variants}
        self.dev = {v: runner.to_device(self.host[v]) for v in self.variants}
        dt = self.dev[self.variants[0]]["q"].dtype
        self.outs = {v: torch.empty(wl.B, wl.T, wl.H, wl.dv, dtype=dt, device="cuda")
                     for v in self.variants}
        self.finals = {v: torch.empty(wl.B, wl.H, wl.dk, wl.dv, device="cuda")
                       for v in self.variants}
        self.auxf = {}
        for v in self.variants:
            shp = aux_shape(v, wl.B, wl.H, wl.dk)
            self.auxf[v] = None if shp is None else torch.empty(*shp, device="cuda")
        wss = [runner.workspace_for(self.dev[v]) for v in self.variants]
        self.ws = max((w for w in wss if w is not None), key=lambda w: w.numel(), default=None)
        dtype_id = dr.DR_BF16 if wl.dtype == "bf16" else dr.DR_FP32
        self.paths = {v: dr.dr_chunk_fwd_path(dr.VARIANT_IDS[v], dtype_id, wl.dk, wl.dv,
                                              wl.chunk) for v in self.variants}

    def call(self, v, stream):
        self.runner.chunk_fwd(self.dev[v], out=self.outs[v], final_state=self.finals[v],
                              aux_final=self.auxf[v], stream=stream, workspace=self.ws)

    def launches_per_step(self, nsm):
        wl = self.wl
        NC = -(-wl.T // wl.chunk)
        return sum(kernels_per_call(self.paths[v], v, wl.B, wl.H, self.ws is not None, nsm, NC)
                   for v in self.variants)

    def time(self, steps, warmup, stream, flush, on_step_start=None):
        """Per variant, the CUDA-event time of each of ``steps`` forwards (L2 flushed
        before every step, outside the events); returns ({variant: [ms]}, [step ms])."""
        torch = self.torch
        for _ in range(max(3, warmup)):
            for v in self.variants:
                self.call(v, stream)
        torch.cuda.synchronize()
        self.dr.check(self.dr.dr_get_device_status(), f"{self.wl.name} warm-up")
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        ev = [(E(), E()) for _ in range(steps)]
        vev = {v: [(E(), E()) for _ in range(steps)] for v in self.variants}
        if on_step_start:
            on_step_start()
        torch.cuda.synchronize()
        for i in range(steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            for v in self.variants:
                vev[v][i][0].record(stream)
                self.call(v, stream)
                vev[v][i][1].record(stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        self.dr.check(self.dr.dr_get_device_status(), f"{self.wl.name} timed")
        return ({v: [s.elapsed_time(e) for s, e in vev[v]] for v in self.variants},
                [s.elapsed_time(e) for s, e in ev])

    def parity_jobs(self, n_pairs):
        """Oracle jobs for sampled (b, h) rows of every variant (CPU inputs)."""
        jobs = []
        for v in self.variants:
            for b, h in sampled_pairs(self.wl.B, self.wl.H, n_pairs):
                jobs.append(((self.wl.name, v, b, h), slice_row(self.host[v], b, h), v, None,
                             None))
        return jobs

    def parity(self, results):
        """max rel. error of the GPU's last outputs against the oracle rows."""
        worst = {"out": 0.0, "state": 0.0, "aux": 0.0}
        for (name, v, b, h), o, S, aux in results:
            if name != self.wl.name:
                continue
            worst["out"] = max(worst["out"], rel_err(
                self.outs[v][b, :, h].double().cpu().numpy(), o[0, :, 0]))
            worst["state"] = max(worst["state"], rel_err(
                self.finals[v][b, h].double().cpu().numpy(), S[0, 0]))
            if aux is not None and self.auxf[v] is not None:
                worst["aux"] = max(worst["aux"], rel_err(
                    self.auxf[v][b, h].double().cpu().numpy(), aux[0, 0]))
        return worst


def forward_entry(fw, var_ms, pk, launches):
    """Per-workload record: mean time per variant, tokens/s, bytes, roofline fraction."""
    wl = fw.wl
    per = {}
    for v in fw.variants:
        ms = statistics.mean(var_ms[v])
        byt = fwd_bytes(wl, v)
        path = fw.paths[v]
        kname = "chunk_" + path
        per[v] = {"ms": ms, "ms_median": statistics.median(var_ms[v]),
                  "tokens_per_s": wl.B * wl.T / (ms / 1e3), "algorithmic_bytes": byt,
                  "gbs": byt / (ms / 1e3) / 1e9, "frac": byt / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                  "path": path, "traffic": measured_traffic(kname, wl.name, v)}
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "d": wl.dk, "chunk": wl.chunk,
            "dtype": wl.dtype, "variants": per, "launches_per_step": launches}


BWD_GRADS = ("dq", "dk", "dv", "dlog_alpha", "deta", "dS0")


def bwd_grad_names(variant):
    """The gradients the bench checks per variant (per token or per row)."""
    if variant in ("kdn", "ikdn"):
        return ("dq", "dk", "dv", "dlog_alpha", "dS0", "domega", "dr")
    return BWD_GRADS + (("dalphaP", "dbetaP") if variant in ("pgdn", "pkda") else ())


def time_backward(torch, dr, runner, fw, steps, stream, flush, pk, pool_submit, n_pairs=2):
    """dr_chunk_bwd on a forward workload's inputs (every variant it lists that the
    backward supports): CUDA-event time per call, L2 flushed between calls; oracle
    jobs for two sampled (b, h) rows per variant.  Returns (entry, gpu rows)."""
    wl = fw.wl
    gen = torch.Generator().manual_seed(wl.seed + 500)
    dO = torch.randn(wl.B, wl.T, wl.H, wl.dv, generator=gen).to(fw.host[fw.variants[0]]["q"].dtype)
    dS = 0.1 * torch.randn(wl.B, wl.H, wl.dk, wl.dv, generator=gen)
    S0 = 0.3 * torch.randn(wl.B, wl.H, wl.dk, wl.dv, generator=gen)
    dOd, dSd, S0d = dO.cuda(), dS.cuda(), S0.cuda()
    entry, rows = {"workload": wl.name, "variants": {}}, {}
    pairs = sampled_pairs(wl.B, wl.H, n_pairs)
    for v in fw.variants:
        ws = runner.bwd_workspace_for(fw.dev[v]) if v in BWD_VARIANTS else None
        if ws is None:
            continue
        grads = runner.chunk_bwd(fw.dev[v], dOd, d_final_state=dSd, init_state=S0d,
                                 workspace=ws, stream=stream)
        for _ in range(2):
            runner.chunk_bwd(fw.dev[v], dOd, d_final_state=dSd, init_state=S0d, workspace=ws,
                             stream=stream, grads=grads)
        torch.cuda.synchronize()
        dr.check(dr.dr_get_device_status(), "backward warm-up")
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        ev = [(E(), E()) for _ in range(steps)]
        for i in range(steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            runner.chunk_bwd(fw.dev[v], dOd, d_final_state=dSd, init_state=S0d, workspace=ws,
                             stream=stream, grads=grads)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        dr.check(dr.dr_get_device_status(), "backward")
        ms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in ev)
        byt = bwd_bytes(wl, v)
        nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        entry["variants"][v] = {"ms": ms, "tokens_per_s": wl.B * wl.T / (ms / 1e3),
                                "algorithmic_bytes": byt, "gbs": byt / (ms / 1e3) / 1e9,
                                "frac": byt / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                                "launches_per_call": bwd_kernels_per_call(v, wl.B, wl.H, nsm)}
        names = bwd_grad_names(v)
        for b, h in pairs:
            rows[(wl.name, v, b, h)] = {n: (grads[n][b, h] if n == "dS0" else grads[n][b, :, h])
                                        .double().cpu().numpy() for n in names}
            pool_submit([((wl.name, v, b, h), slice_row(fw.host[v], b, h), v,
                          dO[b:b + 1, :, h:h + 1].float().numpy(),
                          dS[b:b + 1, h:h + 1].numpy(), S0[b:b + 1, h:h + 1].numpy())])
        del ws
    entry["parity_sample"] = f"{len(pairs)} (b, h) rows per variant"
    entry["kernels"] = ("forward prep + carry (saving chunk-start states and E), reverse "
                        "carry, per-chunk state products, per-chunk local gradients")
    return entry, rows


def decode_setup(torch, runner, W, wl, variant, n_pool=8):
    """Device inputs for n_pool decode steps, a state and the gain state."""
    steps = [W.generate_decode_step(wl, s, variant) for s in range(n_pool)]
    g = torch.Generator().manual_seed(wl.seed + 77)
    S0 = 0.05 * torch.randn(wl.B, wl.H, wl.dk, wl.dv, generator=g)
    shp = aux_shape(variant, wl.B, wl.H, wl.dk)
    aux0 = None
    if variant in ("pgdn", "pkda"):
        aux0 = torch.rand(*shp, generator=g)
    elif variant in ("kdn", "ikdn"):
        aux0 = 0.5 + torch.rand(*shp, generator=g)
    elif variant == "ekdn":
        aux0 = torch.eye(wl.dk).expand(*shp).contiguous()
    return steps, S0, aux0


def time_decode(torch, dr, runner, W, wl, variant, n_steps, stream, pk):
    steps, S0, aux0 = decode_setup(torch, runner, W, wl, variant)
    dsteps = [runner.to_device(s) for s in steps]
    S = S0.cuda()
    aux = None if aux0 is None else aux0.cuda()
    dt = dsteps[0]["q"].dtype
    dout = torch.empty(wl.B, wl.H, wl.dv, dtype=dt, device="cuda")
    for i in range(5):
        runner.decode_step(dsteps[i % len(dsteps)], S, aux, out=dout, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n_steps):
        runner.decode_step(dsteps[i % len(dsteps)], S, aux, out=dout, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    dr.check(dr.dr_get_device_status(), f"decode {variant}")
    ms = e0.elapsed_time(e1) / n_steps
    db = decode_bytes(wl, variant)
    gbs = db / (ms / 1e3) / 1e9
    kernel = "kalman" if variant == "ekdn" else "decode"
    return {"workload": wl.name, "variant": variant, "B": wl.B, "H": wl.H, "d": wl.dk,
            "ms_per_step": ms, "gbs": gbs, "frac": gbs / pk["hbm_gbs"],
            "algorithmic_bytes_per_step": db, "steps": n_steps,
            "traffic": measured_traffic(kernel, wl.name), "tokens_per_s": wl.B / (ms / 1e3),
            "launches": n_steps, "kernel": kernel}


def decode_parity(torch, runner, W, wl, variant, n_steps, pairs):
    """Decode n_steps from a seeded state on the full batch; returns the GPU's
    outputs and final state for the sampled rows, and the oracle jobs for them."""
    steps, S0, aux0 = decode_setup(torch, runner, W, wl, variant, n_pool=n_steps)
    S = S0.cuda()
    aux = None if aux0 is None else aux0.cuda()
    outs = [runner.decode_step(runner.to_device(s), S, aux).clone() for s in steps]
    torch.cuda.synchronize()
    gpu = {(b, h): (torch.stack([o[b, h] for o in outs]).double().cpu().numpy(),
                    S[b, h].double().cpu().numpy()) for b, h in pairs}
    jobs = []
    for b, h in pairs:
        seq = {}
        for k, t in steps[0].items():
            if not hasattr(t, "numpy"):
                seq[k] = t
            elif k == "mu":
                seq[k] = t[h:h + 1].float().numpy()
            else:
                seq[k] = torch.stack([s[k][b:b + 1, h:h + 1] for s in steps], 1).float().numpy()
        s0 = S0[b:b + 1, h:h + 1].numpy()
        a0 = None if aux0 is None else aux0[b:b + 1, h:h + 1].numpy()
        jobs.append((("decode", variant, b, h), seq, variant, s0, a0))
    return gpu, jobs


# ---------------------------------------------------------------- our arm

def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)

    # the oracle pool must exist before the first CUDA call (spawn context anyway)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    pool = None
    want_oracle = rank == 0 and world == 1 and not (args.no_cpu_baseline and args.no_configs)
    if want_oracle:
        pool = mp.get_context("spawn").Pool(min(os.cpu_count() or 1, 16))

    import torch
    from recurrent_associative_memory_gb300 import dr, runner
    from recurrent_associative_memory_gb300 import workloads as W

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    pk = peaks()
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    parity_async = []   # pending oracle jobs (AsyncResult), collected at the end

    def submit(jobs):
        if pool is not None and not args.no_configs:
            parity_async.append(pool.map_async(_oracle_parity, jobs, chunksize=1))

    bwd_async = []

    def submit_bwd(jobs):
        if pool is not None and not args.no_configs:
            bwd_async.append(pool.map_async(_oracle_bwd_parity, jobs, chunksize=1))

    # ---------------- headline workload: the timed region
    wl = W.WORKLOADS[args.workload]
    head = Forward(torch, dr, runner, W, wl)
    variants = head.variants
    submit(head.parity_jobs(2))
    clocks = ClockSampler(local)

    def start_clocks():
        clocks.start()
        time.sleep(0.25)
        barrier(world)

    var_ms, step_ms = head.time(args.steps, args.warmup, stream, flush, start_clocks)
    barrier(world)
    clk = clocks.stop()
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    launches = args.steps * head.launches_per_step(nsm)
    value = job_tokens_per_s(world, args.steps, len(variants), wl.B, wl.T, total_s)
    entry = forward_entry(head, var_ms, pk, head.launches_per_step(nsm))
    dom = max(variants, key=lambda v: entry["variants"][v]["ms"])
    dv_ = entry["variants"][dom]
    kname = "chunk_" + dv_["path"]
    kdesc = f"{kname} ({dom})"
    if dv_["path"] == "tc_split":
        kdesc = f"{kname}: chunk_prep + chunk_carry of one dr_chunk_fwd call ({dom})"
    roof = {"bound": "hbm", "achieved": dv_["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": dv_["frac"], "traffic": dv_["traffic"], "kernel": kdesc,
            "algorithmic_bytes_per_launch": dv_["algorithmic_bytes"],
            "peak_source": pk["src"]}
    result = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
              "steps": args.steps, "warmup": max(3, args.warmup),
              "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
              "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.dk,
                         "dv": wl.dv, "chunk": wl.chunk, "variants": variants,
                         "state": "fp32", "l2": "flushed between timed steps (256 MiB write)",
                         "parallelism": f"replicas x{world}"},
              "roofline": roof, "variants": entry["variants"], "gpu_launches": launches,
              "clocks": clk}
    configs = {}

    # ---------------- the backward (GDN and KLA) on the headline workload
    bwd_rows, bwd_entries = {}, {}
    if not args.no_backward:
        bent, rows_ = time_backward(torch, dr, runner, head, min(args.steps, 20), stream,
                                    flush, pk, submit_bwd)
        if bent["variants"]:
            bwd_entries[bent["workload"]] = bent
            bwd_rows.update(rows_)
        torch.cuda.empty_cache()

    # ---------------- every configuration's workload, timed the same way
    if not args.no_configs:
        for tag, name in CONFIG_WORKLOADS:
            if name == "kla_decode_bf16":
                continue
            if name == wl.name:
                configs[tag] = dict(entry, parity=None)
                configs[tag]["_fw"] = head
                continue
            fw = Forward(torch, dr, runner, W, W.WORKLOADS[name])
            submit(fw.parity_jobs(1 if fw.wl.T > 16384 else 2))
            vms, _ = fw.time(min(args.steps, 20), 3, stream, flush)
            configs[tag] = forward_entry(fw, vms, pk, fw.launches_per_step(nsm))
            configs[tag]["_fw"] = fw
            if not args.no_backward and ("pgdn" in fw.variants or "kdn" in fw.variants):
                # PGDN's and Diagonal KDN's backward too
                bent, rows_ = time_backward(torch, dr, runner, fw, min(args.steps, 10), stream,
                                            flush, pk, submit_bwd, n_pairs=1)
                if bent["variants"]:
                    bwd_entries[bent["workload"]] = bent
                    bwd_rows.update(rows_)
                torch.cuda.empty_cache()
            # keep only what the parity check reads; free the rest of the device memory
            fw.dev = fw.ws = None
            torch.cuda.empty_cache()

    # ---------------- the rows beyond the configurations (KDA, PKDA, isotropic KDN,
    #                  exact Kalman): forward, and the backward where it exists
    next_rows = {}
    if not args.no_configs and not args.no_next:
        for tag, name in NEXT_WORKLOADS:
            fw = Forward(torch, dr, runner, W, W.WORKLOADS[name])
            submit(fw.parity_jobs(1))
            vms, _ = fw.time(min(args.steps, 10), 3, stream, flush)
            next_rows[tag] = forward_entry(fw, vms, pk, fw.launches_per_step(nsm))
            next_rows[tag]["_fw"] = fw
            if not args.no_backward and any(v in BWD_VARIANTS for v in fw.variants):
                bent, rows_ = time_backward(torch, dr, runner, fw, min(args.steps, 10), stream,
                                            flush, pk, submit_bwd, n_pairs=1)
                if bent["variants"]:
                    bwd_entries[bent["workload"]] = bent
                    bwd_rows.update(rows_)
                torch.cuda.empty_cache()
            fw.dev = fw.ws = None
            torch.cuda.empty_cache()

    # ---------------- decode step (batch 256, H 16): HBM GB/s, every variant
    dec_parity = None
    if not args.no_decode:
        dwl = W.WORKLOADS["kla_decode_bf16"]
        result["decode"] = time_decode(torch, dr, runner, W, dwl, "kla", args.decode_steps,
                                       stream, pk)
        per_var = {}
        for v, base in DECODE_VARIANTS.items():
            vwl = W.small(base, B=dwl.B, T=1, H=dwl.H, seed=dwl.seed)
            per_var[v] = time_decode(torch, dr, runner, W, vwl, v,
                                     max(10, args.decode_steps // 4), stream, pk)
        result["decode"]["variants"] = per_var
        if not args.no_configs:
            pairs = [(0, 0), (dwl.B // 2, dwl.H // 2), (dwl.B - 1, dwl.H - 1)]
            gpu, jobs = decode_parity(torch, runner, W, dwl, "kla", 16, pairs)
            submit(jobs)
            dec_parity = gpu
            configs["4b"] = {"workload": dwl.name, "B": dwl.B, "H": dwl.H, "d": dwl.dk,
                             "ms_per_step": result["decode"]["ms_per_step"],
                             "tokens_per_s": result["decode"]["tokens_per_s"],
                             "algorithmic_bytes": result["decode"]["algorithmic_bytes_per_step"],
                             "gbs": result["decode"]["gbs"], "frac": result["decode"]["frac"],
                             "traffic": result["decode"]["traffic"],
                             "parity_sample": f"{len(pairs)} (b, h) rows x 16 steps from a "
                                              "seeded state"}

    # ---------------- end to end through the public API with pinned host buffers
    if not args.no_e2e:
        dev, outs, finals, auxf, ws = head.dev, head.outs, head.finals, head.auxf, head.ws
        host = head.host
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
        dr.check(dr.dr_get_device_status(), "e2e")
        sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
        result["e2e"] = {"value": world * n * len(variants) * wl.B * wl.T / sec, "unit": "tokens/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}
        # the last e2e step wrote set (n - 1) & 1; point the parity check at it
        head.outs = osets[(n - 1) & 1]

    # ---------------- parity of every timed configuration against the oracle
    if parity_async:
        results = [r for a in parity_async for r in a.get()]
        for tag, c in configs.items():
            fw = c.pop("_fw", None)
            if fw is not None:
                c["parity"] = fw.parity(results)
                c["parity_sample"] = (f"{len(sampled_pairs(fw.wl.B, fw.wl.H, 2))} (b, h) rows "
                                      "per variant" if fw.wl.T <= 16384 else
                                      "1 (b, h) row")
        for tag, c in next_rows.items():
            fw = c.pop("_fw", None)
            if fw is not None:
                c["parity"] = fw.parity(results)
                c["parity_sample"] = "1 (b, h) row"
        if dec_parity is not None:
            worst = {"out": 0.0, "state": 0.0}
            for (name, v, b, h), o, S, _ in results:
                if name == "decode":
                    go, gS = dec_parity[(b, h)]
                    worst["out"] = max(worst["out"], rel_err(go, o[0, :, 0]))
                    worst["state"] = max(worst["state"], rel_err(gS, S[0, 0]))
            configs["4b"]["parity"] = worst
    if bwd_entries:
        result["backward"] = {"workloads": bwd_entries}
    if bwd_async and bwd_entries:
        worst = {}
        for a_ in bwd_async:
            for tag, ref in a_.get():
                gpu = bwd_rows[tag]
                ent = bwd_entries[tag[0]].setdefault("parity", {})
                for n, r_ in ref.items():
                    r = r_[0, 0] if n == "dS0" else r_[0, :, 0]
                    e = rel_err(gpu[n], r)
                    worst[n] = max(worst.get(n, 0.0), e)
                    ent[n] = max(ent.get(n, 0.0), e)
        result["backward"]["parity"] = worst
    for c in list(configs.values()) + list(next_rows.values()):
        c.pop("_fw", None)
    if next_rows:
        result["next_rows"] = next_rows
    if configs:
        result["configs"] = configs
        result["parity_bar"] = {"bf16": 5e-3, "fp32": 1e-4,
                                "measure": "max|gpu - oracle| / max|oracle|"}

    # ---------------- the oracle on the host cores (warm pool)
    if pool is not None and not args.no_cpu_baseline:
        n_heads = min(args.cpu_sample_heads, wl.H)
        oracle_sample(args.workload, n_heads, pool)          # warm: inputs drawn per worker
        tok, secs, cpu_s, cores = oracle_sample(args.workload, n_heads, pool,
                                                reps=args.cpu_sample_reps)
        one = oracle_one_core(args.workload, pool)
        result["cpu_baseline"] = {"value": tok / secs, "unit": "tokens/s", "cores": cores,
                                  "kind": "oracle", "cpu_seconds": cpu_s, "wall_seconds": secs,
                                  "one_core_value": one,
                                  "sample": cpu_sample_text(wl, n_heads, args.cpu_sample_reps)}
    if pool is not None:
        pool.close()
        pool.join()
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
