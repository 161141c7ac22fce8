"""Call the library on a workload's tensors: output allocation + marshalling.

``chunk_fwd`` and ``decode_step`` take the dict produced by ``workloads``
(already on the GPU), allocate the outputs with torch and call
``dr.dr_chunk_fwd`` / ``dr.dr_decode_step``.  They do no arithmetic of their
own.
"""

from __future__ import annotations

import torch

from . import dr

GATE_KEYS = ("log_alpha", "eta", "alphaP", "betaP", "mu", "omega", "r")


def to_device(inp: dict, device="cuda") -> dict:
    """Copy every tensor of an input dict to ``device`` (contiguous)."""
    return {k: (v.to(device).contiguous() if torch.is_tensor(v) else v) for k, v in inp.items()}


def params_for(inp: dict, aux_init=None, aux_final=None, check_finite=False) -> dr.DrParams:
    dtype = dr.DR_BF16 if inp["q"].dtype == torch.bfloat16 else dr.DR_FP32
    return dr.make_params(dtype=dtype, q_l2norm=inp.get("q_l2norm", False),
                          k_l2norm=inp.get("k_l2norm", False), eta=inp.get("eta"),
                          alphaP=inp.get("alphaP"), betaP=inp.get("betaP"), mu=inp.get("mu"),
                          x=inp.get("x", 1.5), log_floor=inp.get("log_floor", 1e-12),
                          omega=inp.get("omega"), r=inp.get("r"),
                          info_scale=inp.get("info_scale", 1.0), aux_init=aux_init,
                          aux_final=aux_final, check_finite=check_finite)


def workspace_for(inp: dict, chunk=None):
    """Device scratch for dr_chunk_fwd on these inputs (None where no path uses one)."""
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dtype = dr.DR_BF16 if q.dtype == torch.bfloat16 else dr.DR_FP32
    n = dr.dr_chunk_fwd_workspace_bytes(dr.VARIANT_IDS[inp["variant"]], dtype, B, T, H, dk,
                                        v.shape[-1], chunk or inp.get("chunk", 64))
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def chunk_fwd(inp: dict, *, init_state=None, aux_init=None, chunk=None, want_final=True,
              check_finite=False, stream=None, out=None, final_state=None, aux_final=None,
              workspace="auto"):
    """Run dr_chunk_fwd on a device input dict; returns (out, final_state, aux_final).

    ``workspace``: "auto" allocates the scratch the fastest path wants, None runs
    without one, or a uint8 device tensor to reuse."""
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    variant = dr.VARIANT_IDS[inp["variant"]]
    if isinstance(workspace, str):
        workspace = workspace_for(inp, chunk)
    if out is None:
        out = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if want_final and final_state is None:
        final_state = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    if want_final and aux_final is None and inp["variant"] in ("pgdn", "kdn", "pkda"):
        aux_final = torch.empty(B, H, dk, dtype=torch.float32, device=q.device)
    if want_final and aux_final is None and inp["variant"] == "ikdn":   # one variance per head
        aux_final = torch.empty(B, H, dtype=torch.float32, device=q.device)
    if want_final and aux_final is None and inp["variant"] == "ekdn":   # dense covariance
        aux_final = torch.empty(B, H, dk, dk, dtype=torch.float32, device=q.device)
    p = params_for(inp, aux_init=aux_init, aux_final=aux_final, check_finite=check_finite)
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    st = dr.dr_chunk_fwd(q, k, v, inp["log_alpha"], p, variant, inp.get("eps", 1e-6), init_state,
                         out, final_state, B, T, H, dk, dv, chunk or inp.get("chunk", 64), stream)
    dr.check(st, "dr_chunk_fwd")
    return out, final_state, aux_final


def decode_step(inp: dict, state, aux_state=None, out=None, stream=None, check_finite=False):
    """One dr_decode_step on [B, H, d] device inputs; state/aux updated in place."""
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, H, dk = k.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    p = params_for(inp, check_finite=check_finite)
    st = dr.dr_decode_step(q, k, v, inp["log_alpha"], p, dr.VARIANT_IDS[inp["variant"]],
                           inp.get("eps", 1e-6), state, aux_state, out, B, H, dk, dv, stream)
    dr.check(st, "dr_decode_step")
    return out


def bwd_workspace_for(inp: dict, chunk=None):
    """Device scratch for dr_chunk_bwd on these inputs (None where unsupported)."""
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dtype = dr.DR_BF16 if q.dtype == torch.bfloat16 else dr.DR_FP32
    n = dr.dr_chunk_bwd_workspace_bytes(dr.VARIANT_IDS[inp["variant"]], dtype, B, T, H, dk,
                                        v.shape[-1], chunk or inp.get("chunk", 64))
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def chunk_bwd(inp: dict, d_out, *, d_final_state=None, init_state=None, aux_init=None,
              d_aux_final=None, want_dS0=True, chunk=None, stream=None, workspace="auto",
              grads=None):
    """Run dr_chunk_bwd on a device input dict; returns a dict of fp32 gradients
    (dq, dk, dv, dlog_alpha, deta, with want_dS0 dS0, and for PGDN / PKDA dalphaP,
    dbetaP, dmu, daux0; Diagonal / isotropic KDN domega, dr, daux0 and no deta).
    With per-channel decay (KDA, PKDA, KDN, isotropic KDN) dlog_alpha is [B,T,H,dk].  ``grads`` may hold
    preallocated output tensors under the same names."""
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if isinstance(workspace, str):
        workspace = bwd_workspace_for(inp, chunk)
    f32 = dict(dtype=torch.float32, device=q.device)
    g = dict(grads or {})
    g.setdefault("dq", torch.empty(B, T, H, dk, **f32))
    g.setdefault("dk", torch.empty(B, T, H, dk, **f32))
    g.setdefault("dv", torch.empty(B, T, H, dv, **f32))
    per_channel = inp["variant"] in ("kda", "kdn", "pkda", "ikdn")
    g.setdefault("dlog_alpha", torch.empty(*((B, T, H, dk) if per_channel else (B, T, H)), **f32))
    if inp["variant"] not in ("kdn", "ikdn"):
        g.setdefault("deta", torch.empty(B, T, H, **f32))
    if want_dS0:
        g.setdefault("dS0", torch.empty(B, H, dk, dv, **f32))
    if inp["variant"] in ("pgdn", "pkda"):
        g.setdefault("dalphaP", torch.empty(B, T, H, **f32))
        g.setdefault("dbetaP", torch.empty(B, T, H, **f32))
        g.setdefault("dmu", torch.empty(H, **f32))
        g.setdefault("daux0", torch.empty(B, H, dk, **f32))
    if inp["variant"] == "kdn":
        g.setdefault("domega", torch.empty(B, T, H, dk, **f32))
        g.setdefault("dr", torch.empty(B, T, H, **f32))
        g.setdefault("daux0", torch.empty(B, H, dk, **f32))
    if inp["variant"] == "ikdn":   # one variance per head: omega per token
        g.setdefault("domega", torch.empty(B, T, H, **f32))
        g.setdefault("dr", torch.empty(B, T, H, **f32))
        g.setdefault("daux0", torch.empty(B, H, **f32))
    p = params_for(inp, aux_init=aux_init)
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    gs = dr.make_grads(dq=g["dq"], dk=g["dk"], dv=g["dv"], d_log_alpha=g["dlog_alpha"],
                       d_eta=g.get("deta"), d_init_state=g.get("dS0"), d_alphaP=g.get("dalphaP"),
                       d_betaP=g.get("dbetaP"), d_mu=g.get("dmu"), d_aux_init=g.get("daux0"),
                       d_aux_final=d_aux_final, d_omega=g.get("domega"), d_r=g.get("dr"))
    st = dr.dr_chunk_bwd(q, k, v, inp["log_alpha"], p, dr.VARIANT_IDS[inp["variant"]],
                         inp.get("eps", 1e-6), init_state, d_out, d_final_state, gs, B, T, H, dk,
                         dv, chunk or inp.get("chunk", 64), stream)
    dr.check(st, "dr_chunk_bwd")
    return g
