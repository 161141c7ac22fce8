"""CUDA-graph capture of the library's calls (include/dr.h: calls are asynchronous
on their stream and may be captured).

After one eager call per path (first-call set-up happens outside capture), a
forward on each tensor-core path and a decode step are captured into one
graph; the graph is replayed on new input contents written into the same
buffers and must match eager calls on those inputs bit for bit.
"""

import pytest
import torch

from recurrent_associative_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _fill(dst: dict, src: dict):
    for k, v in src.items():
        if torch.is_tensor(v):
            dst[k].copy_(v)


def test_forward_and_decode_replay_from_a_cuda_graph():
    from recurrent_associative_memory_gb300 import dr, runner

    def inputs(variant, seed):
        wl = W.small("pgdn_bf16" if variant == "pgdn" else "gdn_kla_bf16", B=2, T=200, H=3,
                     seed=seed)
        return W.generate(wl, variant)

    variants = ["kla", "pgdn"]
    dev = {v: runner.to_device(inputs(v, 11)) for v in variants}
    ws = {v: runner.workspace_for(dev[v]) for v in variants}
    nows = {"kla": None}                                  # also the no-workspace path
    dstep = runner.to_device(W.generate_decode_step(W.small("kla_decode_bf16", B=8, H=4), 0))
    state0 = torch.randn(8, 4, 128, 128, device="cuda") * 0.05

    def outputs():
        o = {v: torch.empty_like(dev[v]["v"]) for v in variants}
        o["kla_nows"] = torch.empty_like(dev["kla"]["v"])
        S = {k: torch.empty(2, 3, 128, 128, device="cuda") for k in o}
        aux = torch.empty(2, 3, 128, device="cuda")
        return o, S, aux

    def run(o, S, aux, state, dout, stream=None):
        for v in variants:
            runner.chunk_fwd(dev[v], out=o[v], final_state=S[v],
                             aux_final=aux if v == "pgdn" else None, workspace=ws[v],
                             stream=stream)
        runner.chunk_fwd(dev["kla"], out=o["kla_nows"], final_state=S["kla_nows"],
                         workspace=nows["kla"], stream=stream)
        runner.decode_step(dstep, state, out=dout, stream=stream)

    # eager warm-up on the capture stream
    side = torch.cuda.Stream()
    og, Sg, auxg = outputs()
    state_g = state0.clone()
    dout_g = torch.empty(8, 4, 128, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(side):
        run(og, Sg, auxg, state_g, dout_g)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(og, Sg, auxg, state_g, dout_g)

    for seed in (12, 13):   # new contents in the captured buffers, then replay
        for v in variants:
            _fill(dev[v], inputs(v, seed))
        _fill(dstep, W.generate_decode_step(W.small("kla_decode_bf16", B=8, H=4), seed))
        state_g.copy_(state0)
        graph.replay()
        torch.cuda.synchronize()
        oe, Se, auxe = outputs()
        state_e = state0.clone()
        dout_e = torch.empty_like(dout_g)
        run(oe, Se, auxe, state_e, dout_e)
        torch.cuda.synchronize()
        assert dr.dr_get_device_status() == 0
        for k in oe:
            assert torch.equal(og[k], oe[k]) and torch.equal(Sg[k], Se[k]), (seed, k)
        assert torch.equal(auxg, auxe)
        assert torch.equal(dout_g, dout_e) and torch.equal(state_g, state_e)


def test_chained_prep_and_exact_kalman_replay_from_a_cuda_graph():
    """The CUDA-core two-phase path with the variance handed between prep tasks
    (a memset of its flags and ticket counter, then ticket-ordered tasks) and the
    exact Kalman decode step (state and covariance in place), captured and
    replayed on new contents: every replay resets the chain, and the results
    equal eager calls bit for bit."""
    from recurrent_associative_memory_gb300 import dr, runner

    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    wl_k = W.small("kdn_bf16", B=2, T=64 * 3 + 5, H=26)
    assert 3 * wl_k.B * wl_k.H >= nsm                     # the chained prep
    wl_a = W.small("kda_bf16", B=2, T=100, H=3)
    wl_e = W.small("ekdn_bf16", B=4, T=1, H=3)

    def inputs(seed):
        return {"kdn": W.generate(wl_k, "kdn", seed=seed), "kda": W.generate(wl_a, "kda", seed=seed)}

    def estep(seed):
        return W.generate_decode_step(wl_e, seed, "ekdn")

    dev = {v: runner.to_device(x) for v, x in inputs(31).items()}
    ws = {v: runner.workspace_for(dev[v]) for v in dev}
    dstep = runner.to_device(estep(31))
    g = torch.Generator().manual_seed(5)
    A = torch.randn(4, 3, 128, 128, generator=g, dtype=torch.float64)
    P0 = (A @ A.transpose(-1, -2) / 128 + 0.5 * torch.eye(128, dtype=torch.float64)).float().cuda()
    S0 = (0.05 * torch.randn(4, 3, 128, 128, generator=g)).cuda()

    def outputs():
        o = {v: torch.empty_like(dev[v]["v"]) for v in dev}
        S = {v: torch.empty(dev[v]["k"].shape[0], dev[v]["k"].shape[2], 128, 128, device="cuda")
             for v in dev}
        p = torch.empty(2, 26, 128, device="cuda")
        return o, S, p

    def run(o, S, p, state, cov, dout, stream=None):
        for v in dev:
            runner.chunk_fwd(dev[v], out=o[v], final_state=S[v],
                             aux_final=p if v == "kdn" else None, workspace=ws[v], stream=stream)
        runner.decode_step(dstep, state, cov, out=dout, stream=stream)

    side = torch.cuda.Stream()
    og, Sg, pg = outputs()
    state_g, cov_g = S0.clone(), P0.clone()
    dout_g = torch.empty(4, 3, 128, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(side):
        run(og, Sg, pg, state_g, cov_g, dout_g)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(og, Sg, pg, state_g, cov_g, dout_g)

    for seed in (32, 33):
        for v, x in inputs(seed).items():
            _fill(dev[v], x)
        _fill(dstep, estep(seed))
        state_g.copy_(S0)
        cov_g.copy_(P0)
        graph.replay()
        torch.cuda.synchronize()
        oe, Se, pe = outputs()
        state_e, cov_e = S0.clone(), P0.clone()
        dout_e = torch.empty_like(dout_g)
        run(oe, Se, pe, state_e, cov_e, dout_e)
        torch.cuda.synchronize()
        assert dr.dr_get_device_status() == 0
        for v in oe:
            assert torch.equal(og[v], oe[v]) and torch.equal(Sg[v], Se[v]), (seed, v)
        assert torch.equal(pg, pe)
        assert torch.equal(dout_g, dout_e) and torch.equal(state_g, state_e)
        assert torch.equal(cov_g, cov_e)
