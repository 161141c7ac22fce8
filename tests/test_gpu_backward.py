"""GPU parity of the backward (dr_chunk_bwd) against the fp64 oracle's reverse sweep.

Every gradient -- dq, dk, dv, d log alpha, d eta and dL/dS_0; for PGDN also
d alphaP, d betaP, d mu and dL/dA_0 -- of L = <dO, O> + <dS_T, S_T> (PGDN:
+ <dA_T, A_T>) is compared element by element with
``oracle.backward.tokenwise_backward`` on the same seeded bf16 inputs (the
oracle upcasts the rounded values), at sizes with several chunks and a ragged
tail, with and without the L2 norms and the initial state, and at the GDN/KLA
workload's full size on sampled (b, h) rows.  Bar: max|gpu - ref| / max|ref|
<= 5e-3 (the bf16 bar of the forward).
"""

import numpy as np
import pytest
import torch

from oracle import backward as obw
from parity_util import TOL, np64, rel_err, slice_heads
from recurrent_associative_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dlog_alpha", "deta", "dS0")


@pytest.fixture(scope="module")
def rt():
    from recurrent_associative_memory_gb300 import dr, runner
    return dr, runner


PG_NAMES = ("dalphaP", "dbetaP", "dmu", "daux0")


KDN_NAMES = ("dq", "dk", "dv", "dlog_alpha", "dS0", "domega", "dr", "daux0")


def oracle_grads(inp, dO, dS, S0, aux0=None, daux=None):
    f = lambda t: None if t is None else t.double().cpu().numpy()  # noqa: E731
    g = obw.tokenwise_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_alpha"]),
                               inp["variant"], f(dO), f(dS), eta=f(inp.get("eta")),
                               eps=inp["eps"], q_l2norm=inp["q_l2norm"],
                               k_l2norm=inp["k_l2norm"], S0=f(S0),
                               alphaP=f(inp.get("alphaP")), betaP=f(inp.get("betaP")),
                               mu=f(inp.get("mu")), x=inp.get("x", 1.5),
                               log_floor=inp.get("log_floor", 1e-12), omega=f(inp.get("omega")),
                               r=f(inp.get("r")), info_scale=inp.get("info_scale", 1.0),
                               aux0=f(aux0), daux_T=f(daux))
    if inp["variant"] in ("kdn", "ikdn"):
        return {n: g[n] for n in KDN_NAMES}
    names = NAMES + (PG_NAMES if inp["variant"] in ("pgdn", "pkda") else ())
    return {n: g[n] for n in names}


def run_case(rt, inp, seed=0, with_state=True, with_dS=True):
    dr, runner = rt
    B, T, H, dk = inp["k"].shape
    gen = torch.Generator().manual_seed(seed)
    dO = torch.randn(B, T, H, 128, generator=gen).to(inp["q"].dtype)
    dS = 0.1 * torch.randn(B, H, 128, 128, generator=gen) if with_dS else None
    S0 = 0.3 * torch.randn(B, H, 128, 128, generator=gen) if with_state else None
    dev = runner.to_device(inp)
    g = runner.chunk_bwd(dev, dO.cuda(), d_final_state=None if dS is None else dS.cuda(),
                         init_state=None if S0 is None else S0.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    return g, dO, dS, S0


def check(g, ref, pairs=None, tol=TOL["bf16"]):
    errs = {}
    for n in ref:
        x = g[n]
        if pairs is not None:
            x = torch.stack([x[b, h] if n == "dS0" else x[b, :, h] for b, h in pairs])
            x = x[:, None] if n == "dS0" else x[:, :, None]
        errs[n] = rel_err(np64(x), ref[n])
    assert all(e <= tol for e in errs.values()), errs
    return errs


@pytest.mark.parametrize("variant", ["gdn", "kla"])
@pytest.mark.parametrize("T,norms", [(64, True), (200, True), (333, False), (1, True)])
def test_backward_matches_oracle(rt, variant, T, norms):
    wl = W.small("pgdn_bf16" if norms else "gdn_kla_bf16", variants=("gdn", "kla"), B=2, T=T,
                 H=3, seed=50 + T)
    inp = W.generate(wl, variant)
    g, dO, dS, S0 = run_case(rt, inp, seed=T)
    check(g, oracle_grads(inp, dO, dS, S0))


@pytest.mark.parametrize("variant", ["gdn", "kla"])
def test_backward_without_state_or_final_gradient(rt, variant):
    wl = W.small("gdn_kla_bf16", B=1, T=130, H=2, seed=9)
    inp = W.generate(wl, variant)
    g, dO, dS, S0 = run_case(rt, inp, seed=4, with_state=False, with_dS=False)
    check(g, oracle_grads(inp, dO, dS, S0))


@pytest.mark.parametrize("variant", ["gdn", "kla"])
def test_backward_workload_full_size_sampled(rt, variant):
    """B8 H8 T2048 (the GDN/KLA workload, raw keys): sampled (b, h) rows against
    the oracle on those rows (heads are independent)."""
    wl = W.WORKLOADS["gdn_kla_bf16"]
    inp = W.generate(wl, variant)
    g, dO, dS, S0 = run_case(rt, inp, seed=11)
    pairs = [(0, 0), (wl.B - 1, wl.H - 1)]
    sub = slice_heads(inp, pairs)
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    dS_s = torch.stack([dS[b, h] for b, h in pairs])[:, None]
    S0_s = torch.stack([S0[b, h] for b, h in pairs])[:, None]
    check(g, oracle_grads(sub, dO_s, dS_s, S0_s), pairs=pairs)


def test_backward_is_deterministic_and_reuses_its_workspace(rt):
    dr, runner = rt
    wl = W.small("gdn_kla_bf16", B=2, T=150, H=2, seed=3)
    dev = runner.to_device(W.generate(wl, "kla"))
    gen = torch.Generator().manual_seed(1)
    dO = torch.randn(2, 150, 2, 128, generator=gen).to(torch.bfloat16).cuda()
    ws = runner.bwd_workspace_for(dev)
    g1 = {k: v.clone() for k, v in runner.chunk_bwd(dev, dO, workspace=ws).items()}
    ws.fill_(255)                                   # garbage left in the workspace
    g2 = runner.chunk_bwd(dev, dO, workspace=ws)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n


@pytest.mark.parametrize("T,norms", [(200, True), (333, True), (130, False)])
def test_pgdn_backward_matches_oracle(rt, T, norms):
    """PGDN: the memory part as GDN with the record's explicit write keys, then the
    key statistic's adjoint carried backwards over the whole row (d beta, d alphaP,
    d betaP, d mu, dL/dA_0 and the key gradient through B(A)); a nonzero A_0 and
    dL/dA_T."""
    dr, runner = rt
    wl = W.small("pgdn_bf16", B=2, T=T, H=3, seed=70 + T, k_l2norm=norms)
    inp = W.generate(wl, "pgdn")
    B, H = 2, 3
    gen = torch.Generator().manual_seed(T)
    dO = torch.randn(B, T, H, 128, generator=gen).to(torch.bfloat16)
    dS = 0.1 * torch.randn(B, H, 128, 128, generator=gen)
    S0 = 0.3 * torch.randn(B, H, 128, 128, generator=gen)
    A0 = torch.rand(B, H, 128, generator=gen) * 2.0
    dA = 0.1 * torch.randn(B, H, 128, generator=gen)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda(), d_final_state=dS.cuda(),
                         init_state=S0.cuda(), aux_init=A0.cuda(), d_aux_final=dA.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    check(g, oracle_grads(inp, dO, dS, S0, A0, dA))


def test_pgdn_backward_workload_sampled(rt):
    """B4 H16 T4096 (the PGDN workload): the per-token gradients of sampled rows
    against the oracle on those rows."""
    dr, runner = rt
    wl = W.WORKLOADS["pgdn_bf16"]
    inp = W.generate(wl, "pgdn")
    gen = torch.Generator().manual_seed(12)
    dO = torch.randn(wl.B, wl.T, wl.H, 128, generator=gen).to(torch.bfloat16)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    pairs = [(0, 5), (wl.B - 1, 5)]
    sub = slice_heads(inp, pairs)
    sub["mu"] = sub["mu"][:1]          # both rows are head 5: the slice has one head
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    ref = oracle_grads(sub, dO_s, None, None)
    for n in ("dmu", "daux0", "dS0"):   # per head / per row: checked on the small cases
        ref.pop(n)
    errs = {}
    for n, r in ref.items():
        x = torch.stack([g[n][b, :, h] for b, h in pairs])
        x = x[:, :, None]
        errs[n] = rel_err(np64(x), r)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


# ------------------------------------------------------------ per-channel decay (KDA)

@pytest.mark.parametrize("T,norms", [(64, True), (200, True), (333, False), (1, True), (130, True)])
def test_kda_backward_matches_oracle(rt, T, norms):
    """KDA (w = eta k^, D = diag(alpha) per channel): the sub-chunk-referenced
    Gram gradients, the per-channel decay gradient [B,T,H,dk], d eta, dL/dS_0."""
    wl = W.small("kda_bf16", B=2, T=T, H=3, seed=90 + T, k_l2norm=norms, q_l2norm=norms)
    inp = W.generate(wl, "kda")
    g, dO, dS, S0 = run_case(rt, inp, seed=T)
    assert g["dlog_alpha"].shape == (2, T, 3, 128)
    check(g, oracle_grads(inp, dO, dS, S0))


def test_kda_backward_many_rows_chained_shape(rt):
    """Enough rows that the forward's per-channel prep runs its chunk-major order
    (3 B H >= SM count), a ragged tail."""
    dr, runner = rt
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    H = -(-nsm // 6)
    wl = W.small("kda_bf16", B=2, T=150, H=H, seed=7)
    inp = W.generate(wl, "kda")
    g, dO, dS, S0 = run_case(rt, inp, seed=3)
    pairs = [(0, 0), (1, H - 1)]
    sub = slice_heads(inp, pairs)
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    dS_s = torch.stack([dS[b, h] for b, h in pairs])[:, None]
    S0_s = torch.stack([S0[b, h] for b, h in pairs])[:, None]
    check(g, oracle_grads(sub, dO_s, dS_s, S0_s), pairs=pairs)


def test_kda_backward_workload_sampled(rt):
    """B4 H16 T8192 (the KDA workload): one sampled row's per-token gradients."""
    dr, runner = rt
    wl = W.WORKLOADS["kda_bf16"]
    inp = W.generate(wl, "kda")
    gen = torch.Generator().manual_seed(13)
    dO = torch.randn(wl.B, wl.T, wl.H, 128, generator=gen).to(torch.bfloat16)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    pairs = [(wl.B - 1, 7)]
    sub = slice_heads(inp, pairs)
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    ref = oracle_grads(sub, dO_s, None, None)
    ref.pop("dS0")
    errs = {}
    for n, r in ref.items():
        x = torch.stack([g[n][b, :, h] for b, h in pairs])[:, :, None]
        errs[n] = rel_err(np64(x), r)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


# ------------------------------------------------------------ Diagonal KDN

def run_kdn(rt, inp, seed, with_aux=True):
    dr, runner = rt
    B, T, H, dk = inp["k"].shape
    gen = torch.Generator().manual_seed(seed)
    dO = torch.randn(B, T, H, 128, generator=gen).to(torch.bfloat16)
    dS = 0.1 * torch.randn(B, H, 128, 128, generator=gen)
    S0 = 0.3 * torch.randn(B, H, 128, 128, generator=gen)
    p0 = (0.5 + torch.rand(B, H, 128, generator=gen)) if with_aux else None
    dp = (0.1 * torch.randn(B, H, 128, generator=gen)) if with_aux else None
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda(), d_final_state=dS.cuda(),
                         init_state=S0.cuda(), aux_init=None if p0 is None else p0.cuda(),
                         d_aux_final=None if dp is None else dp.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    return g, dO, dS, S0, p0, dp


@pytest.mark.parametrize("T,norms", [(64, True), (200, True), (333, False), (1, True)])
def test_kdn_backward_matches_oracle(rt, T, norms):
    """Diagonal KDN: the chunk part as KDA with the Kalman gains as write vectors,
    then the variance adjoint carried backwards over the row (d omega, d r, the key
    gradient through the gain and the variance update, the decay gradient through
    alpha^2 p, dL/dp_0), with a nonzero p_0 and dL/dp_T."""
    wl = W.small("kdn_bf16", B=2, T=T, H=3, seed=110 + T, k_l2norm=norms, q_l2norm=norms)
    inp = W.generate(wl, "kdn")
    g, dO, dS, S0, p0, dp = run_kdn(rt, inp, seed=T)
    assert "deta" not in g and g["domega"].shape == (2, T, 3, 128)
    check(g, oracle_grads(inp, dO, dS, S0, aux0=p0, daux=dp))


def test_kdn_backward_information_scale_and_default_variance(rt):
    """mu = d_k (the information-scaled update) and p_0 = 1 (no aux_init)."""
    wl = W.small("kdn_bf16", B=1, T=150, H=2, seed=5, info_scale=128.0)
    inp = W.generate(wl, "kdn")
    g, dO, dS, S0, p0, dp = run_kdn(rt, inp, seed=6, with_aux=False)
    check(g, oracle_grads(inp, dO, dS, S0))


def test_kdn_backward_many_rows_chained_shape(rt):
    """Enough rows for the forward's chained variance hand-over (3 B H >= SMs)."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    H = -(-nsm // 6)
    wl = W.small("kdn_bf16", B=2, T=150, H=H, seed=8)
    inp = W.generate(wl, "kdn")
    g, dO, dS, S0, p0, dp = run_kdn(rt, inp, seed=9)
    pairs = [(0, 1), (1, H - 1)]
    sub = slice_heads(inp, pairs)
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    dS_s = torch.stack([dS[b, h] for b, h in pairs])[:, None]
    S0_s = torch.stack([S0[b, h] for b, h in pairs])[:, None]
    p0_s = torch.stack([p0[b, h] for b, h in pairs])[:, None]
    dp_s = torch.stack([dp[b, h] for b, h in pairs])[:, None]
    ref = oracle_grads(sub, dO_s, dS_s, S0_s, aux0=p0_s, daux=dp_s)
    errs = {}
    for n, r in ref.items():
        if n in ("dS0", "daux0"):
            x = torch.stack([g[n][b, h] for b, h in pairs])[:, None]
        else:
            x = torch.stack([g[n][b, :, h] for b, h in pairs])[:, :, None]
        errs[n] = rel_err(np64(x), r)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


def test_kdn_backward_workload_sampled(rt):
    """B4 H16 T8192 (the Diagonal KDN workload): one sampled row's per-token gradients."""
    dr, runner = rt
    wl = W.WORKLOADS["kdn_bf16"]
    inp = W.generate(wl, "kdn")
    gen = torch.Generator().manual_seed(14)
    dO = torch.randn(wl.B, wl.T, wl.H, 128, generator=gen).to(torch.bfloat16)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    pairs = [(1, 9)]
    sub = slice_heads(inp, pairs)
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    ref = oracle_grads(sub, dO_s, None, None)
    for n in ("dS0", "daux0"):
        ref.pop(n)
    errs = {}
    for n, r in ref.items():
        x = torch.stack([g[n][b, :, h] for b, h in pairs])[:, :, None]
        errs[n] = rel_err(np64(x), r)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


# ------------------------------------------------------------ PKDA, isotropic KDN

@pytest.mark.parametrize("T,norms", [(200, True), (333, False), (64, True)])
def test_pkda_backward_matches_oracle(rt, T, norms):
    """PKDA: KDA's chunk part with the PGDN write keys, then the key statistic's
    adjoint (d beta, d alphaP, d betaP, d mu, dL/dA_0); nonzero A_0 and dL/dA_T."""
    dr, runner = rt
    wl = W.small("pkda_bf16", B=2, T=T, H=3, seed=130 + T, k_l2norm=norms)
    inp = W.generate(wl, "pkda")
    B, H = 2, 3
    gen = torch.Generator().manual_seed(T)
    dO = torch.randn(B, T, H, 128, generator=gen).to(torch.bfloat16)
    dS = 0.1 * torch.randn(B, H, 128, 128, generator=gen)
    S0 = 0.3 * torch.randn(B, H, 128, 128, generator=gen)
    A0 = torch.rand(B, H, 128, generator=gen) * 2.0
    dA = 0.1 * torch.randn(B, H, 128, generator=gen)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda(), d_final_state=dS.cuda(),
                         init_state=S0.cuda(), aux_init=A0.cuda(), d_aux_final=dA.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    check(g, oracle_grads(inp, dO, dS, S0, aux0=A0, daux=dA))


@pytest.mark.parametrize("T,norms", [(200, True), (333, False), (1, True)])
def test_ikdn_backward_matches_oracle(rt, T, norms):
    """Isotropic KDN: the chunk part with w = beta k^, then the head variance's
    scalar adjoint (d omega and d r per token, d log alpha through the mean squared
    decay, the key gradient through beta and ||k^||^2, dL/db_0)."""
    wl = W.small("ikdn_bf16", B=2, T=T, H=3, seed=150 + T, k_l2norm=norms)
    inp = W.generate(wl, "ikdn")
    dr, runner = rt
    B, H = 2, 3
    gen = torch.Generator().manual_seed(T)
    dO = torch.randn(B, T, H, 128, generator=gen).to(torch.bfloat16)
    dS = 0.1 * torch.randn(B, H, 128, 128, generator=gen)
    S0 = 0.3 * torch.randn(B, H, 128, 128, generator=gen)
    b0 = 0.5 + torch.rand(B, H, generator=gen)
    db = 0.1 * torch.randn(B, H, generator=gen)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda(), d_final_state=dS.cuda(),
                         init_state=S0.cuda(), aux_init=b0.cuda(), d_aux_final=db.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    check(g, oracle_grads(inp, dO, dS, S0, aux0=b0, daux=db))


@pytest.mark.parametrize("variant", ["pkda", "ikdn"])
def test_gain_variants_backward_many_rows_chained_shape(rt, variant):
    """Enough rows for the forward's chained hand-over of the gain state."""
    dr, runner = rt
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    H = -(-nsm // 6)
    wl = W.small(f"{variant}_bf16", B=2, T=150, H=H, seed=17)
    inp = W.generate(wl, variant)
    gen = torch.Generator().manual_seed(2)
    dO = torch.randn(2, 150, H, 128, generator=gen).to(torch.bfloat16)
    g = runner.chunk_bwd(runner.to_device(inp), dO.cuda())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    pairs = [(0, H - 1), (1, H - 1)]   # one head: the slice keeps PKDA's mu per head
    sub = slice_heads(inp, pairs)
    if variant == "pkda":
        sub["mu"] = sub["mu"][:1]
    dO_s = torch.stack([dO[b, :, h] for b, h in pairs])[:, :, None]
    ref = oracle_grads(sub, dO_s, None, None)
    for n in ("dS0", "daux0", "dmu"):
        ref.pop(n, None)
    errs = {}
    for n, r in ref.items():
        x = torch.stack([g[n][b, :, h] for b, h in pairs])[:, :, None]
        errs[n] = rel_err(np64(x), r)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
