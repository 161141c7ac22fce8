"""GPU: the device-side give-up path of a bounded wait, and a long decode chain.

* A wait that runs out.  The chained prep of the per-channel-decay two-phase
  path hands each row's gain state from one chunk's task to the next through a
  flag in the workspace.  The test-only hook makes the task that would raise one
  flag skip it and shortens the wait to 10 ms, so the next chunk's task waits on
  a flag that nothing sets: the call must come back with DR_ERR_TIMEOUT through
  dr_get_device_status() within a bounded time (no trap, no hang), and the next
  call on the same context must be right again.
* The 64K-token KLA prefill followed by 4096 in-place decode steps at batch 256
  x 16 heads, the prefill state replicated into every batch row (the prefill's
  B = 1 against the decode's batch 256).  The oracle runs the same prefill on
  two heads and the same decode steps: three sampled rows over all 4096 steps,
  and every batch row of those two heads over the first 16 steps.
"""

import time

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, np64, rel_err, run_oracle
from recurrent_associative_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt():
    from recurrent_associative_memory_gb300 import dr, runner
    return dr, runner


@pytest.mark.parametrize("variant", ["kdn", "pkda"])
def test_chained_prep_wait_gives_up_on_a_withheld_flag(rt, variant):
    dr, runner = rt
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    B, T = 2, 256
    H = -(-nsm // (3 * B))            # 3 B H >= SM count: the chained prep runs
    assert 3 * B * H >= nsm
    NC = -(-T // 64)
    base = {"kdn": "kdn_bf16", "pkda": "pkda_bf16"}[variant]
    inp = W.generate(W.small(base, B=B, T=T, H=H, seed=41), variant)
    dev = runner.to_device(inp)
    assert dr.dr_chunk_fwd_path(dr.VARIANT_IDS[variant], dr.DR_BF16, 128, 128, 64) == "tc_pc_split"
    flag = (1 * H + 2) * NC + 2       # row (b = 1, h = 2), the hand-over into chunk 2
    assert dr.dr_get_device_status() == 0
    try:
        assert dr.dr_set_chain_fault_for_testing(flag, 10_000_000) == 0
        t0 = time.perf_counter()
        runner.chunk_fwd(dev)
        st = dr.dr_get_device_status()
        elapsed = time.perf_counter() - t0
    finally:
        assert dr.dr_set_chain_fault_for_testing(-1, 2_000_000_000) == 0
    assert st == dr.DR_ERR_TIMEOUT, dr.STATUS.get(st, st)
    assert elapsed < 1.5
    assert dr.dr_get_device_status() == 0          # read once, cleared
    # the context is still usable, and the next call is right
    out, S, aux = runner.chunk_fwd(dev)
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    pairs = [(1, 2), (0, 0)]
    o_ref, S_ref, aux_ref = run_oracle(inp, pairs=pairs)
    o = torch.stack([out[b, :, h] for b, h in pairs])[:, :, None]
    Sg = torch.stack([S[b, h] for b, h in pairs])[:, None]
    ag = torch.stack([aux[b, h] for b, h in pairs])[:, None]
    assert rel_err(np64(o), o_ref) <= TOL["bf16"]
    assert rel_err(np64(Sg), S_ref) <= TOL["bf16"]
    assert rel_err(np64(ag), aux_ref) <= TOL["bf16"]


def test_hook_refuses_bad_arguments(rt):
    dr, _ = rt
    assert dr.dr_set_chain_fault_for_testing(-2, 1000) == dr.DR_ERR_ARG
    assert dr.dr_set_chain_fault_for_testing(-1, 0) == dr.DR_ERR_ARG


def _oracle_row_prefill(inp, h):
    """fp64 prefill of head h of a B = 1 workload: the final state [dk, dv]."""
    _, S, _ = run_oracle(inp, pairs=[(0, h)])
    return S[0, 0]


def _draw(gen, shape, key, dtype):
    """Seeded decode inputs with the GDN/KLA workload's distributions."""
    if key in ("q", "v"):
        return torch.randn(shape, generator=gen).to(dtype)
    if key == "k":
        x = torch.randn(shape, generator=gen)
        return (x * torch.exp(0.5 * torch.randn(shape[:-1] + (1,), generator=gen))).to(dtype)
    if key == "eta":
        return torch.sigmoid(torch.randn(shape, generator=gen))
    if key == "log_alpha":
        return -torch.nn.functional.softplus(torch.randn(shape, generator=gen) + 2.0)
    raise KeyError(key)


def test_prefill_then_4096_decode_steps_at_batch_256(rt):
    dr, runner = rt
    pwl = W.WORKLOADS["kla_prefill_bf16"]
    dwl = W.WORKLOADS["kla_decode_bf16"]
    n_steps, n_all = 4096, 16
    pre = W.generate(pwl, "kla")
    _, S_pre, _ = runner.chunk_fwd(runner.to_device(pre))
    S = S_pre.expand(dwl.B, -1, -1, -1).contiguous()          # replicated into every row
    heads = [0, dwl.H - 1]
    rows = [(0, heads[0]), (dwl.B // 2, heads[1]), (dwl.B - 1, heads[0])]

    # Per-step inputs: a pool of 32 seeded full-batch steps; over the first 16
    # steps fresh seeded inputs for every batch row of the two checked heads; and
    # fresh seeded inputs for the three sampled rows at every step.
    pool = [W.generate_decode_step(dwl, s) for s in range(32)]
    keys = ("q", "k", "v", "eta", "log_alpha")
    g = torch.Generator().manual_seed(4242)
    dt = pool[0]["q"].dtype
    rows_in = {k: _draw(g, (n_steps, len(rows)) + tuple(pool[0][k].shape[2:]), k, dt) for k in keys}
    all_in = {k: _draw(g, (n_all, dwl.B, len(heads)) + tuple(pool[0][k].shape[2:]), k, dt)
              for k in keys}
    for i, (b, h) in enumerate(rows):     # the sampled rows keep their own sequence
        for k in keys:
            all_in[k][:, b, heads.index(h)] = rows_in[k][:n_all, i]
    dpool = [runner.to_device(p) for p in pool]
    d_rows = {k: v.cuda() for k, v in rows_in.items()}
    d_all = {k: v.cuda() for k, v in all_in.items()}
    hidx = torch.tensor(heads, device="cuda")
    bsel = torch.tensor([b for b, _ in rows], device="cuda")
    hsel = torch.tensor([h for _, h in rows], device="cuda")
    outs_rows, outs_all = [], []
    step = {k: v.clone() if torch.is_tensor(v) else v for k, v in dpool[0].items()}
    for s in range(n_steps):
        for k in keys:
            step[k].copy_(dpool[s % 32][k])
            if s < n_all:
                step[k][:, hidx] = d_all[k][s]
            else:
                step[k][bsel, hsel] = d_rows[k][s]
        o = runner.decode_step(step, S)
        outs_rows.append(o[bsel, hsel])
        if s < n_all:
            outs_all.append(o[:, hidx].clone())
    torch.cuda.synchronize()
    assert dr.dr_get_device_status() == 0
    o_rows = torch.stack(outs_rows, 1).double().cpu().numpy()       # [3, steps, dv]
    o_all = torch.stack(outs_all, 1).double().cpu().numpy()         # [B, 16, 2, dv]

    # oracle: the same prefill on the two heads, then the same decode inputs
    S0 = {h: _oracle_row_prefill(pre, h) for h in heads}
    f = lambda t: t.double().numpy()  # noqa: E731
    kw = dict(eps=dwl.eps, q_l2norm=dwl.q_l2norm, k_l2norm=dwl.k_l2norm)
    for i, (b, h) in enumerate(rows):
        q, k, v, eta, la = (f(rows_in[n][:, i])[None, :, None] for n in keys)
        o_ref, S_ref, _ = oracle.tokenwise(q, k, v, la, "kla", eta=eta, S0=S0[h][None, None], **kw)
        assert rel_err(o_rows[i], o_ref[0, :, 0]) <= TOL["bf16"], (b, h)
        assert rel_err(S[b, h].double().cpu().numpy(), S_ref[0, 0]) <= TOL["bf16"], (b, h)
    for j, h in enumerate(heads):
        q, k, v, eta, la = (np.swapaxes(f(all_in[n][:, :, j]), 0, 1)[:, :, None] for n in keys)
        S0b = np.broadcast_to(S0[h], (dwl.B, 1) + S0[h].shape).copy()
        o_ref, _, _ = oracle.tokenwise(q, k, v, la, "kla", eta=eta, S0=S0b, **kw)
        assert rel_err(o_all[:, :, j], o_ref[:, :, 0]) <= TOL["bf16"], h
