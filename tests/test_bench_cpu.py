"""Host-side pieces of the benchmark, on CPU: the algorithmic byte counts the
roofline divides by (per head-token: q, k, v, o and the gates; plus the final
state), the decode step's bytes, and the rule that a recorded DRAM traffic
figure is only used for the kernel source it was captured on."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from recurrent_associative_memory_gb300 import workloads as W  # noqa: E402


# q, k, v, o bf16 (1024) + fp32 gates: log alpha, eta (GDN/KLA); + alphaP, betaP
# (PGDN); per-channel log alpha and omega + r (KDN); per-channel log alpha + eta
# (KDA), + alphaP, betaP (PKDA)
@pytest.mark.parametrize("variant,per_head_token", [("gdn", 1032), ("kla", 1032),
                                                     ("pgdn", 1040), ("kdn", 2052),
                                                     ("kda", 1540), ("pkda", 1548),
                                                     ("ikdn", 1544), ("ekdn", 2052)])
def test_forward_bytes_per_head_token(variant, per_head_token):
    name = {"gdn": "gdn_kla_bf16", "kla": "gdn_kla_bf16", "pgdn": "pgdn_bf16",
            "kdn": "kdn_bf16", "kda": "kda_bf16", "pkda": "pkda_bf16",
            "ikdn": "ikdn_bf16", "ekdn": "ekdn_bf16"}[variant]
    wl = W.WORKLOADS[name]
    ht = wl.B * wl.T * wl.H
    extra = wl.H * 4 if variant in ("pgdn", "pkda") else 0     # the per-head mu
    assert bench.fwd_bytes(wl, variant, with_final=False) == ht * per_head_token + extra


def test_bench_workload_bytes():
    wl = W.WORKLOADS["gdn_kla_bf16"]
    state = wl.B * wl.H * wl.dk * wl.dv * 4
    assert bench.fwd_bytes(wl, "kla") == 8 * 2048 * 8 * 1032 + state == 139_460_608


def test_decode_step_bytes():
    wl = W.WORKLOADS["kla_decode_bf16"]
    # per (b, h): fp32 state read + write, q, k, v, o in bf16, two fp32 gates
    per_bh = 2 * 128 * 128 * 4 + 4 * 128 * 2 + 8
    assert bench.decode_bytes(wl) == wl.B * wl.H * per_bh == 541_097_984


def test_recorded_traffic_is_tied_to_the_kernel_source(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["chunk_tc_split"]
    fake_root = tmp_path
    os.makedirs(fake_root / "profiles")
    stale = dict(rec, source_sha256="0" * 64)
    (fake_root / "profiles" / "traffic.json").write_text(json.dumps({"chunk_tc_split": stale}))
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "f" * 64)
    assert bench.measured_traffic("chunk_tc_split", rec["workload"], "kla") is None
    fresh = dict(rec, source_sha256="f" * 64)
    (fake_root / "profiles" / "traffic.json").write_text(json.dumps({"chunk_tc_split": fresh}))
    assert bench.measured_traffic("chunk_tc_split", rec["workload"], "kla") == rec["dram_bytes_per_launch"]
    assert bench.measured_traffic("chunk_tc_split", "pgdn_bf16", "pgdn") is None   # other workload


def test_default_arguments_are_one_gpu_and_short(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    args = bench.parse()
    assert args.gpus == 1 and args.impl == "ours" and args.workload == "gdn_kla_bf16"
    assert args.warmup >= 3 and 1 <= args.steps <= 200


def test_kernels_per_call_counts_every_path():
    """The gpu_launches claim: kernels per dr_chunk_fwd call by path and variant."""
    k = bench.kernels_per_call
    assert k("tc_split", "kla", 8, 8, True, 152) == 2          # prep + carry
    assert k("tc_split", "pgdn", 4, 16, True, 152) == 4        # + statistic map and scan
    assert k("tc_split", "kla", 8, 8, False, 152) == 1         # no workspace: one kernel
    assert k("tc_ws", "kla", 8, 8, False, 152) == 1
    assert k("tc_pc_split", "kdn", 4, 16, True, 152) == 2      # variance chained in the prep
    assert k("tc_pc_split", "kdn", 1, 2, True, 152) == 4       # few rows: map + scan first
    assert k("tc_pc_split", "kda", 1, 2, True, 152) == 2       # no gain state across chunks
    assert k("tc_pc_split", "pkda", 1, 2, True, 152) == 1      # few rows: the fused kernel
    assert k("tc_pc_split", "ikdn", 4, 16, True, 152) == 2
    assert k("simt_split", "kdn", 4, 16, True, 152) == 2       # fp32: CUDA-core prep
    assert k("kalman", "ekdn", 4, 16, False, 152) == 1
    assert k("simt", "kla", 1, 2, False, 152) == 1
    # few long rows: segment-parallel carry, + segment composition + replay pass
    assert k("tc_split", "kla", 1, 16, True, 152, 1024) == 4
    assert k("tc_split", "pgdn", 1, 16, True, 152, 1024) == 6
    assert k("tc_split", "kla", 8, 8, True, 152, 32) == 2      # 64 rows: one pass
    assert k("tc_split", "kla", 1, 16, True, 152, 4) == 2      # too short to cut in 3


def test_segment_count_rule():
    """Segments per row: G = (SMs / rows - 2) / 4 + 2, shrunk until the
    segments (ceil(NC / G) chunks, at least 2) are all non-empty."""
    s = bench.seg_segments
    assert s(152, 16, 1024) == 3           # 64K-token prefill, 16 heads
    assert s(152, 1, 1024) == 38           # one row: 39 would leave the last one empty
    assert s(152, 26, 1024) == 0           # 6 rows > SMs / 26: one pass
    assert s(152, 2, 7) == 4               # 7 chunks: segments of 2, 2, 2, 1
    assert s(152, 2, 5) == 3               # 2, 2, 1
    assert s(152, 2, 4) == 0               # 3 segments of 2 would leave one empty


@pytest.mark.parametrize("variant,gates,aux", [("gdn", 8, 0), ("pgdn", 16, 128), ("kdn", 1028, 128),
                                               ("kda", 516, 0), ("pkda", 524, 128), ("ikdn", 520, 1),
                                               ("ekdn", 1028, 128 * 128)])
def test_decode_step_bytes_per_variant(variant, gates, aux):
    """Each variant's decode step moves its state and gain state twice (read, write),
    q, k, v, o once and its own gates; PGDN / PKDA also read the per-head mu."""
    wl = W.small("kla_decode_bf16", B=4, H=3)
    per_bh = 2 * (128 * 128 + aux) * 4 + 4 * 128 * 2 + gates
    mu = 3 * 4 if variant in ("pgdn", "pkda") else 0
    assert bench.decode_bytes(wl, variant) == 4 * 3 * per_bh + mu
    shp = bench.aux_shape(variant, 4, 3, 128)
    assert (shp is None) == (aux == 0)
    if shp is not None:
        n = 1
        for s in shp[2:]:
            n *= s
        assert n == aux


def test_every_configuration_has_a_workload():
    tags = [t for t, _ in bench.CONFIG_WORKLOADS]
    assert tags == ["0", "1", "2", "3", "4a", "4b"]
    for _, name in bench.CONFIG_WORKLOADS:
        assert name in W.WORKLOADS
    for v, base in bench.DECODE_VARIANTS.items():
        assert v in W.WORKLOADS[base].variants


def test_parity_row_slice_matches_the_oracle_on_the_full_input():
    """The (b, h) row the bench sends to a pool worker gives the oracle's result for
    that row of the full input (heads are independent)."""
    import numpy as np
    import oracle
    wl = W.small("pgdn_bf16", B=2, T=40, H=3, seed=5)
    inp = W.generate(wl, "pgdn")
    row = bench.slice_row(inp, 1, 2)
    tag, o, S, aux = bench._oracle_parity((("x", "pgdn", 1, 2), row, "pgdn", None, None))
    f = lambda t: t.double().numpy()  # noqa: E731
    o_all, S_all, A_all = oracle.tokenwise(f(inp["q"]), f(inp["k"]), f(inp["v"]),
                                           f(inp["log_alpha"]), "pgdn", eta=f(inp["eta"]),
                                           eps=wl.eps, q_l2norm=wl.q_l2norm,
                                           k_l2norm=wl.k_l2norm, alphaP=f(inp["alphaP"]),
                                           betaP=f(inp["betaP"]), mu=f(inp["mu"]))
    assert np.allclose(o[0, :, 0], o_all[1, :, 2], rtol=0, atol=1e-12)
    assert np.allclose(S[0, 0], S_all[1, 2], rtol=0, atol=1e-12)
    assert np.allclose(aux[0, 0], A_all[1, 2], rtol=0, atol=1e-12)


def test_cpu_baseline_times_only_the_oracle_in_a_warm_pool():
    """oracle_sample counts B*T tokens per variant pass scaled by the heads sampled,
    and after a warm-up call the wall time is close to the workers' own oracle time
    (inputs are drawn once per worker, outside the timed calls)."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(2) as pool:
        bench.oracle_sample("gdn_kla_bf16", 2, pool)
        tok, wall, cpu, cores = bench.oracle_sample("gdn_kla_bf16", 2, pool, reps=2)
        one = bench.oracle_one_core("gdn_kla_bf16", pool)
    wl = W.WORKLOADS["gdn_kla_bf16"]
    assert tok == 2 * 2 * wl.T * 2 / wl.H
    assert cores == 2
    assert cpu <= 2.0 * wall * cores and wall <= 2.0 * cpu
    assert one > 0


def test_backward_bytes():
    """Per head-token: q, k, v, dL/do in bf16 (1024), two fp32 gates (8), dq, dk, dv in
    fp32 (1536), d log alpha and d eta (8); per (b, h): S_0 and dL/dS_T in, dL/dS_0 out."""
    wl = W.WORKLOADS["gdn_kla_bf16"]
    assert bench.bwd_bytes(wl) == wl.B * wl.T * wl.H * 2576 + 3 * wl.B * wl.H * 128 * 128 * 4


def test_backward_parity_row_slice_matches_the_oracle_on_the_full_input():
    import numpy as np
    from oracle import backward as obw
    wl = W.small("gdn_kla_bf16", B=2, T=30, H=2, dk=8, dv=8, seed=6)
    inp = W.generate(wl, "kla")
    g = np.random.default_rng(0)
    dO = g.standard_normal((2, 30, 2, 8))
    dS = g.standard_normal((2, 2, 8, 8))
    S0 = g.standard_normal((2, 2, 8, 8))
    tag, ref = bench._oracle_bwd_parity((("kla", 1, 0), bench.slice_row(inp, 1, 0), "kla",
                                         dO[1:2, :, 0:1], dS[1:2, 0:1], S0[1:2, 0:1]))
    f = lambda t: t.double().numpy()  # noqa: E731
    full = obw.tokenwise_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_alpha"]),
                                  "kla", dO, dS, eta=f(inp["eta"]), eps=wl.eps,
                                  q_l2norm=wl.q_l2norm, k_l2norm=wl.k_l2norm, S0=S0)
    for n in ("dq", "dk", "dv", "dlog_alpha", "deta"):
        assert np.allclose(ref[n][0, :, 0], full[n][1, :, 0], rtol=0, atol=1e-10), n
    assert np.allclose(ref["dS0"][0, 0], full["dS0"][1, 0], rtol=0, atol=1e-10)


def test_backward_bytes_pgdn_and_kernel_counts():
    """PGDN's backward also moves alphaP, betaP in and their gradients out (16 more
    bytes per head-token: 2592), mu / dmu and A_0, dA_T, dA_0; it launches its
    statistic's map and scan, the adjoint's chunk maps, scan and gradients and the
    d mu sum besides the five kernels."""
    wl = W.WORKLOADS["pgdn_bf16"]
    ht = wl.B * wl.T * wl.H
    per_bh = 3 * 128 * 128 * 4 + 3 * 128 * 4
    assert bench.bwd_bytes(wl, "pgdn") == ht * 2592 + wl.B * wl.H * per_bh + 2 * wl.H * 4
    assert bench.bwd_kernels_per_call("kla") == 5 and bench.bwd_kernels_per_call("pgdn") == 11


def test_backward_bytes_and_kernel_counts_per_channel_decay():
    """Per-channel decay: d log alpha per channel (512 bytes in, 512 out); Diagonal
    KDN also omega per channel and r in, their gradients out, and p_0, dL/dp_T in,
    dL/dp_0 out; isotropic KDN one variance per head.  Kernels: the forward again
    (prep and carry; Diagonal KDN with few rows also its variance map and scan),
    the reverse carry, the state products, the local gradients, the gain's adjoint."""
    ht = lambda wl: wl.B * wl.T * wl.H  # noqa: E731
    S3 = lambda wl: 3 * wl.B * wl.H * 128 * 128 * 4  # noqa: E731
    kda, kdn, ikdn = (W.WORKLOADS[n] for n in ("kda_bf16", "kdn_bf16", "ikdn_bf16"))
    base = 1024 + 1536
    assert bench.bwd_bytes(kda, "kda") == ht(kda) * (base + 2 * 516) + S3(kda)
    assert bench.bwd_bytes(kdn, "kdn") == (ht(kdn) * (base + 2 * 1028) + S3(kdn)
                                           + 3 * kdn.B * kdn.H * 128 * 4)
    assert bench.bwd_bytes(ikdn, "ikdn") == (ht(ikdn) * (base + 2 * 520) + S3(ikdn)
                                             + 3 * ikdn.B * ikdn.H * 4)
    k = bench.bwd_kernels_per_call
    assert k("kda", 4, 16) == 5 and k("ikdn", 4, 16) == 8 and k("pkda", 4, 16) == 9
    assert k("kdn", 4, 16, 152) == 8 and k("kdn", 1, 2, 152) == 10
    assert set(bench.bwd_grad_names("kdn")) == {"dq", "dk", "dv", "dlog_alpha", "dS0", "domega",
                                                 "dr"}
    assert "dalphaP" in bench.bwd_grad_names("pkda") and "deta" in bench.bwd_grad_names("kda")
