"""GPU parity of the backward (dr_chunk_bwd) against the fp64 oracle's reverse sweep.

Every gradient -- dq, dk, dv, d log alpha, d eta and dL/dS_0 -- of
L = <dO, O> + <dS_T, S_T> is compared element by element with
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


def oracle_grads(inp, dO, dS, S0):
    f = lambda t: None if t is None else t.double().cpu().numpy()  # noqa: E731
    g = obw.tokenwise_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["log_alpha"]),
                               inp["variant"], f(dO), f(dS), eta=f(inp["eta"]), eps=inp["eps"],
                               q_l2norm=inp["q_l2norm"], k_l2norm=inp["k_l2norm"], S0=f(S0))
    return {"dq": g["dq"], "dk": g["dk"], "dv": g["dv"], "dlog_alpha": g["dlog_alpha"],
            "deta": g["deta"], "dS0": g["dS0"]}


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
    for n in NAMES:
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
