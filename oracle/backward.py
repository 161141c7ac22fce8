"""Reverse-mode gradients of the tokenwise recurrence, fp64 (GDN, KLA, KDA).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The forward is the unified recurrence of ``recurrence.py`` (Kalman Delta
Networks notes, section 1, the displayed equation and the table under it):

    S~_t = D_t S_{t-1},  e_t = v_t - S~_t^T k_t,  S_t = S~_t + w_t e_t^T,  o_t = S_t^T q_t

with D_t = alpha_t I (GDN, KLA) or diag(alpha_t) (KDA), alpha = exp(log_alpha),
and w_t = eta k (GDN, KDA) or eta k / (||k||^2 + eps) (KLA notes Eq. (3)).
Given dL/do_t and dL/dS_T, the reverse sweep walks the tokens backwards with
G = dL/dS_t, applying the chain rule to each line above in reverse order:

    o_t = S_t^T q_t          dS_t += q_t do_t^T,          dq_t = S_t do_t
    S_t = S~_t + w_t e_t^T   dS~_t  = G,  dw_t = G e_t,   de_t = G^T w_t
    e_t = v_t - S~_t^T k_t   dv_t   = de_t,  dS~_t -= k_t de_t^T,  dk_t = -S~_t de_t
    S~_t = D_t S_{t-1}       dS_{t-1} = D_t dS~_t,  d alpha_t = <dS~_t, S_{t-1}>
                             (row-wise for diag(alpha_t)),  d log alpha = alpha d alpha
    w_t = eta k (GDN, KDA)   dk_t += eta dw_t,  d eta_t = k^T dw_t
    w_t = eta k / (s + eps)  dk_t += eta dw_t / (s + eps) - 2 eta (k^T dw_t) k / (s + eps)^2,
                             d eta_t = k^T dw_t / (s + eps),   s = ||k||^2

and, with the L2-normalisation flags, x^ = x / ||x|| gives dx = (dx^ - x^ (x^T dx^)) / ||x||.
The states S_t of the forward are kept (fp64, small test sizes only).
"""

from __future__ import annotations

import numpy as np

GRAD_VARIANTS = ("gdn", "kla", "kda")


def _norm_backward(x_raw, dx_hat):
    """Gradient through x^ = x / ||x|| (the normalisation of the forward)."""
    n = np.sqrt(np.sum(x_raw * x_raw, axis=-1, keepdims=True))
    xh = x_raw / n
    return (dx_hat - xh * np.sum(xh * dx_hat, axis=-1, keepdims=True)) / n


def tokenwise_backward(q, k, v, log_alpha, variant: str, do, dS_T=None, *, eta, eps: float = 1e-6,
                       q_l2norm: bool = False, k_l2norm: bool = False, S0=None):
    """Gradients of sum(do * o) + sum(dS_T * S_T) w.r.t. the forward's inputs.

    Shapes as ``recurrence.tokenwise``: q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha
    [B,T,H] (GDN, KLA) or [B,T,H,dk] (KDA); eta [B,T,H]; do [B,T,H,dv];
    dS_T, S0 [B,H,dk,dv] (None = 0).  Returns a dict with dq, dk, dv,
    dlog_alpha, deta, dS0.
    """
    if variant not in GRAD_VARIANTS:
        raise ValueError(f"no backward for variant {variant!r}")
    f = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    q_raw, k_raw, v, la, eta, do = f(q), f(k), f(v), f(log_alpha), f(eta), f(do)
    B, T, H, dk = k_raw.shape
    dv = v.shape[-1]
    qh = q_raw / np.sqrt(np.sum(q_raw * q_raw, axis=-1, keepdims=True)) if q_l2norm else q_raw
    kh = k_raw / np.sqrt(np.sum(k_raw * k_raw, axis=-1, keepdims=True)) if k_l2norm else k_raw
    per_channel = la.ndim == 4
    alpha = np.exp(la)

    # forward, keeping S_{t-1}, e_t, w_t
    S = np.zeros((B, H, dk, dv)) if S0 is None else f(S0).copy()
    S_prev = np.zeros((T, B, H, dk, dv))
    E = np.zeros((T, B, H, dv))
    Wt = np.zeros((T, B, H, dk))
    for t in range(T):
        S_prev[t] = S
        a_t = alpha[:, t]
        S_tilde = (a_t[..., :, None] if per_channel else a_t[..., None, None]) * S
        kt = kh[:, t]
        if variant == "kla":
            w = (eta[:, t] / (np.sum(kt * kt, axis=-1) + eps))[..., None] * kt
        else:
            w = eta[:, t][..., None] * kt
        e = v[:, t] - np.einsum("bhkv,bhk->bhv", S_tilde, kt)
        S = S_tilde + w[..., :, None] * e[..., None, :]
        E[t], Wt[t] = e, w

    # reverse sweep
    G = np.zeros((B, H, dk, dv)) if dS_T is None else f(dS_T).copy()
    dq = np.zeros_like(qh)
    dk_ = np.zeros_like(kh)
    dv_ = np.zeros_like(v)
    dla = np.zeros_like(la)
    deta = np.zeros_like(eta)
    for t in range(T - 1, -1, -1):
        a_t = alpha[:, t]
        S_tilde = (a_t[..., :, None] if per_channel else a_t[..., None, None]) * S_prev[t]
        e, w, kt, qt = E[t], Wt[t], kh[:, t], qh[:, t]
        S_t = S_tilde + w[..., :, None] * e[..., None, :]
        # o_t = S_t^T q_t
        G = G + qt[..., :, None] * do[:, t][..., None, :]
        dq[:, t] = np.einsum("bhkv,bhv->bhk", S_t, do[:, t])
        # S_t = S~_t + w e^T
        dw = np.einsum("bhkv,bhv->bhk", G, e)
        de = np.einsum("bhkv,bhk->bhv", G, w)
        dSt = G.copy()
        # e = v - S~^T k
        dv_[:, t] = de
        dSt = dSt - kt[..., :, None] * de[..., None, :]
        dk_[:, t] = -np.einsum("bhkv,bhv->bhk", S_tilde, de)
        # w
        if variant == "kla":
            s = np.sum(kt * kt, axis=-1) + eps
            kdw = np.sum(kt * dw, axis=-1)
            dk_[:, t] += (eta[:, t] / s)[..., None] * dw - (2 * eta[:, t] * kdw / s ** 2)[..., None] * kt
            deta[:, t] = kdw / s
        else:
            dk_[:, t] += eta[:, t][..., None] * dw
            deta[:, t] = np.sum(kt * dw, axis=-1)
        # S~ = D S_{t-1}
        if per_channel:
            dalpha = np.sum(dSt * S_prev[t], axis=-1)              # [B,H,dk]
            G = a_t[..., :, None] * dSt
        else:
            dalpha = np.sum(dSt * S_prev[t], axis=(-2, -1))        # [B,H]
            G = a_t[..., None, None] * dSt
        dla[:, t] = a_t * dalpha
    if q_l2norm:
        dq = _norm_backward(q_raw, dq)
    if k_l2norm:
        dk_ = _norm_backward(k_raw, dk_)
    return dict(dq=dq, dk=dk_, dv=dv_, dlog_alpha=dla, deta=deta, dS0=G)
