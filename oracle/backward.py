"""Reverse-mode gradients of the tokenwise recurrence, fp64 (GDN, KLA, KDA, PGDN,
PKDA, Diagonal KDN, isotropic KDN, the exact Kalman memory).

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
The gain states carry their own adjoints backwards:

  PGDN / PKDA (PDN notes Eq. (9)): w = eta (B . k), B = exp(-ln(x) s), s = r/(1+|r|),
      r = ln A - mu (A above the floor), A_t = alphaP A_{t-1} + betaP k.k:
      dB = eta k . dw, ds = -ln(x) B dB, dr = ds/(1+|r|)^2, dA_t += dr / A_t,
      d mu -= sum dr, then dA_{t-1} = alphaP dA_t, d alphaP = A_{t-1}^T dA_t,
      d betaP = (k.k)^T dA_t, dk += 2 betaP k . dA_t.
  Diagonal KDN (KDN notes Eqs. (23)-(30), (60)-(65)): p^ = alpha^2 p + omega,
      kappa = p^ . k / (r + z), z = sum p^ k^2, p_t = p^ / (1 + u p^), u = (mu/r) k.k:
      with c = sum dw . p^ . k and den = r + z,
      dp^ = dw . k / den - c k.k / den^2 + dp_t / (1 + u p^)^2,
      du = -dp_t p^^2 / (1 + u p^)^2,  dk = dw . p^ / den - 2 c p^ . k / den^2 + 2 (mu/r) k . du,
      dr = -c / den^2 - (mu / r^2) sum(k.k du),  d omega = dp^,
      dp_{t-1} = alpha^2 dp^,  d alpha += 2 alpha p dp^.
  Isotropic KDN (KDN notes section 7, Eq. (40)): a = mean alpha^2, b^ = a b + omega,
      beta = b^ / (r + b^ s), s = ||k||^2, w = beta k, b_t = b^ / (1 + u b^),
      u = mu s / (dk r): the scalar adjoint db follows the same pattern, and
      d alpha_i += 2 alpha_i (b db^) / dk.
  Exact Kalman (KDN notes section 2.2): P^ = D P D^T + diag(omega), y = P^ k,
      x = P^T k, den = r + k^T y, w = y / den, P_t = P^ - y x^T / den: dP^ = dP_t
      + dy k^T + k dx^T with dy = dw / den - dP_t x / den + dden k, dx = -dP_t^T y / den,
      dden = y^T dP_t x / den^2 - w^T dw / den, then dP_{t-1} = D dP^ D,
      d alpha_i += sum_j (dP^_ij P_ij + dP^_ji P_ji) alpha_j, d omega = diag(dP^).
The states S_t (and the gain states) of the forward are kept (fp64, small test
sizes only).
"""

from __future__ import annotations

import numpy as np

GRAD_VARIANTS = ("gdn", "kla", "kda", "pgdn", "pkda", "kdn", "ikdn", "ekdn")


def _norm_backward(x_raw, dx_hat):
    """Gradient through x^ = x / ||x|| (the normalisation of the forward)."""
    n = np.sqrt(np.sum(x_raw * x_raw, axis=-1, keepdims=True))
    xh = x_raw / n
    return (dx_hat - xh * np.sum(xh * dx_hat, axis=-1, keepdims=True)) / n


def tokenwise_backward(q, k, v, log_alpha, variant: str, do, dS_T=None, *, eta=None,
                       eps: float = 1e-6, q_l2norm: bool = False, k_l2norm: bool = False,
                       S0=None, alphaP=None, betaP=None, mu=None, x: float = 1.5,
                       log_floor: float = 1e-12, omega=None, r=None, info_scale: float = 1.0,
                       aux0=None, daux_T=None):
    """Gradients of sum(do * o) + sum(dS_T * S_T) + sum(daux_T * aux_T) w.r.t. the
    forward's inputs.

    Shapes as ``recurrence.tokenwise``: q, k [B,T,H,dk]; v [B,T,H,dv]; log_alpha
    [B,T,H] (GDN, KLA, PGDN) or [B,T,H,dk] (KDA, PKDA, KDN); eta, alphaP, betaP,
    r [B,T,H]; omega [B,T,H,dk]; mu [H]; do [B,T,H,dv]; dS_T, S0 [B,H,dk,dv];
    aux0, daux_T [B,H,dk] (None = 0, or p_0 = 1 for KDN).  Returns a dict with
    dq, dk, dv, dlog_alpha, dS0 and the variant's gate gradients (deta; dalphaP,
    dbetaP, dmu, daux0; domega, dr, daux0).
    """
    if variant not in GRAD_VARIANTS:
        raise ValueError(f"no backward for variant {variant!r}")
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)  # noqa: E731
    q_raw, k_raw, v, la, eta, do = f(q), f(k), f(v), f(log_alpha), f(eta), f(do)
    alphaP, betaP, mu, omega, r = f(alphaP), f(betaP), f(mu), f(omega), f(r)
    pstat, kdn = variant in ("pgdn", "pkda"), variant == "kdn"
    ikdn, ekdn = variant == "ikdn", variant == "ekdn"
    B, T, H, dk = k_raw.shape
    dv = v.shape[-1]
    qh = q_raw / np.sqrt(np.sum(q_raw * q_raw, axis=-1, keepdims=True)) if q_l2norm else q_raw
    kh = k_raw / np.sqrt(np.sum(k_raw * k_raw, axis=-1, keepdims=True)) if k_l2norm else k_raw
    per_channel = la.ndim == 4
    alpha = np.exp(la)

    # forward, keeping S_{t-1}, e_t, w_t and the gain states
    S = np.zeros((B, H, dk, dv)) if S0 is None else f(S0).copy()
    S_prev = np.zeros((T, B, H, dk, dv))
    E = np.zeros((T, B, H, dv))
    Wt = np.zeros((T, B, H, dk))
    aux = None
    if pstat:
        aux = np.zeros((B, H, dk)) if aux0 is None else f(aux0).copy()
    elif kdn:
        aux = np.ones((B, H, dk)) if aux0 is None else f(aux0).copy()
    elif ikdn:
        aux = np.ones((B, H)) if aux0 is None else f(aux0).copy()
    elif ekdn:
        aux = (np.broadcast_to(np.eye(dk), (B, H, dk, dk)).copy() if aux0 is None
               else f(aux0).copy())
    aux_prev = np.zeros((T,) + aux.shape) if aux is not None else None
    A_all = np.zeros((T,) + aux.shape) if aux is not None else None   # A_t / p^_t / b^_t / P^_t
    for t in range(T):
        S_prev[t] = S
        a_t = alpha[:, t]
        S_tilde = (a_t[..., :, None] if per_channel else a_t[..., None, None]) * S
        kt = kh[:, t]
        if aux is not None:
            aux_prev[t] = aux
        if variant == "kla":
            w = (eta[:, t] / (np.sum(kt * kt, axis=-1) + eps))[..., None] * kt
        elif pstat:
            aux = alphaP[:, t][..., None] * aux + betaP[:, t][..., None] * kt * kt
            A_all[t] = aux
            rr = np.log(np.maximum(aux, log_floor)) - mu[None, :, None]
            Bs = np.exp(-np.log(x) * rr / (1 + np.abs(rr)))
            w = eta[:, t][..., None] * Bs * kt
        elif ikdn:
            b_hat = np.mean(a_t * a_t, axis=-1) * aux + omega[:, t]
            A_all[t] = b_hat
            sk = np.sum(kt * kt, axis=-1)
            w = (b_hat / (r[:, t] + b_hat * sk))[..., None] * kt
            aux = b_hat / (1 + info_scale * sk / (dk * r[:, t]) * b_hat)
        elif ekdn:
            P_hat = a_t[..., :, None] * aux * a_t[..., None, :] + omega[:, t][..., :, None] * np.eye(dk)
            A_all[t] = P_hat
            y = np.einsum("bhij,bhj->bhi", P_hat, kt)
            xv = np.einsum("bhji,bhj->bhi", P_hat, kt)
            den = r[:, t] + np.sum(kt * y, axis=-1)
            w = y / den[..., None]
            aux = P_hat - y[..., :, None] * xv[..., None, :] / den[..., None, None]
        elif kdn:
            p_hat = a_t * a_t * aux + omega[:, t]
            A_all[t] = p_hat
            w = p_hat * kt / (r[:, t] + np.sum(p_hat * kt * kt, axis=-1))[..., None]
            u = (info_scale / r[:, t])[..., None] * kt * kt
            aux = p_hat / (1 + u * p_hat)
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
    deta = np.zeros((B, T, H)) if eta is not None else None
    daux = (np.zeros(aux.shape) if daux_T is None else f(daux_T).copy()) if aux is not None else None
    dalphaP = np.zeros((B, T, H)) if pstat else None
    dbetaP = np.zeros((B, T, H)) if pstat else None
    dmu = np.zeros(H) if pstat else None
    domega = (np.zeros_like(omega) if (kdn or ikdn or ekdn) else None)
    dr_ = np.zeros((B, T, H)) if (kdn or ikdn or ekdn) else None
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
        dalpha_gain = 0.0
        if variant == "kla":
            s = np.sum(kt * kt, axis=-1) + eps
            kdw = np.sum(kt * dw, axis=-1)
            dk_[:, t] += (eta[:, t] / s)[..., None] * dw - (2 * eta[:, t] * kdw / s ** 2)[..., None] * kt
            deta[:, t] = kdw / s
        elif pstat:
            A = A_all[t]
            rr = np.log(np.maximum(A, log_floor)) - mu[None, :, None]
            Bs = np.exp(-np.log(x) * rr / (1 + np.abs(rr)))
            dB = eta[:, t][..., None] * kt * dw
            dk_[:, t] += eta[:, t][..., None] * Bs * dw
            deta[:, t] = np.sum(Bs * kt * dw, axis=-1)
            drr = -np.log(x) * Bs * dB / (1 + np.abs(rr)) ** 2
            dA = daux + np.where(A > log_floor, drr / A, 0.0)
            dmu -= np.sum(np.where(A > log_floor, drr, 0.0), axis=(0, 2))
            dalphaP[:, t] = np.sum(aux_prev[t] * dA, axis=-1)
            dbetaP[:, t] = np.sum(kt * kt * dA, axis=-1)
            dk_[:, t] += 2 * betaP[:, t][..., None] * kt * dA
            daux = alphaP[:, t][..., None] * dA
        elif ikdn:
            b_hat, rt = A_all[t], r[:, t]
            sk = np.sum(kt * kt, axis=-1)
            den = rt + b_hat * sk
            beta = b_hat / den
            uu = info_scale * sk / (dk * rt)
            q1 = 1 + uu * b_hat
            dbeta = np.sum(kt * dw, axis=-1)
            dk_[:, t] += beta[..., None] * dw
            db_hat = dbeta * rt / den ** 2 + daux / q1 ** 2
            du = -daux * b_hat ** 2 / q1 ** 2
            dsk = -dbeta * b_hat ** 2 / den ** 2 + du * info_scale / (dk * rt)
            dr_[:, t] = -dbeta * b_hat / den ** 2 - du * info_scale * sk / (dk * rt ** 2)
            dk_[:, t] += 2 * dsk[..., None] * kt
            domega[:, t] = db_hat
            a_mean = np.mean(a_t * a_t, axis=-1)
            daux = a_mean * db_hat
            dalpha_gain = 2 * a_t * (aux_prev[t] * db_hat)[..., None] / dk
        elif ekdn:
            P_hat, rt, Pp = A_all[t], r[:, t], aux_prev[t]
            y = np.einsum("bhij,bhj->bhi", P_hat, kt)
            xv = np.einsum("bhji,bhj->bhi", P_hat, kt)
            den = rt + np.sum(kt * y, axis=-1)
            wv = y / den[..., None]
            dden = (np.einsum("bhi,bhij,bhj->bh", y, daux, xv) / den ** 2
                    - np.sum(wv * dw, axis=-1) / den)
            dy = dw / den[..., None] - np.einsum("bhij,bhj->bhi", daux, xv) / den[..., None] \
                + dden[..., None] * kt
            dxv = -np.einsum("bhji,bhj->bhi", daux, y) / den[..., None]
            dr_[:, t] = dden
            dk_[:, t] += (dden[..., None] * y + np.einsum("bhji,bhj->bhi", P_hat, dy)
                          + np.einsum("bhij,bhj->bhi", P_hat, dxv))
            dP_hat = daux + dy[..., :, None] * kt[..., None, :] + kt[..., :, None] * dxv[..., None, :]
            domega[:, t] = np.diagonal(dP_hat, axis1=-2, axis2=-1)
            daux = a_t[..., :, None] * dP_hat * a_t[..., None, :]
            dalpha_gain = (np.einsum("bhij,bhij,bhj->bhi", dP_hat, Pp, a_t)
                           + np.einsum("bhji,bhji,bhj->bhi", dP_hat, Pp, a_t))
        elif kdn:
            p_hat = A_all[t]
            rt = r[:, t]
            den = rt + np.sum(p_hat * kt * kt, axis=-1)
            c = np.sum(dw * p_hat * kt, axis=-1)
            u = (info_scale / rt)[..., None] * kt * kt
            q1 = 1 + u * p_hat
            dp_hat = (dw * kt / den[..., None] - (c / den ** 2)[..., None] * kt * kt
                      + daux / q1 ** 2)
            du = -daux * p_hat ** 2 / q1 ** 2
            dk_[:, t] += (dw * p_hat / den[..., None] - (2 * c / den ** 2)[..., None] * p_hat * kt
                          + 2 * (info_scale / rt)[..., None] * kt * du)
            dr_[:, t] = -c / den ** 2 - info_scale / rt ** 2 * np.sum(kt * kt * du, axis=-1)
            domega[:, t] = dp_hat
            daux = a_t * a_t * dp_hat
            dalpha_gain = 2 * a_t * aux_prev[t] * dp_hat
        else:
            dk_[:, t] += eta[:, t][..., None] * dw
            deta[:, t] = np.sum(kt * dw, axis=-1)
        # S~ = D S_{t-1}
        if per_channel:
            dalpha = np.sum(dSt * S_prev[t], axis=-1) + dalpha_gain   # [B,H,dk]
            G = a_t[..., :, None] * dSt
        else:
            dalpha = np.sum(dSt * S_prev[t], axis=(-2, -1))        # [B,H]
            G = a_t[..., None, None] * dSt
        dla[:, t] = a_t * dalpha
    if q_l2norm:
        dq = _norm_backward(q_raw, dq)
    if k_l2norm:
        dk_ = _norm_backward(k_raw, dk_)
    out = dict(dq=dq, dk=dk_, dv=dv_, dlog_alpha=dla, dS0=G)
    if deta is not None and not (kdn or ikdn or ekdn):
        out["deta"] = deta
    if pstat:
        out.update(dalphaP=dalphaP, dbetaP=dbetaP, dmu=dmu, daux0=daux)
    if kdn or ikdn or ekdn:
        out.update(domega=domega, dr=dr_, daux0=daux)
    return out


def _gain_forward(variant, kh, alpha, *, eta, eps, alphaP, betaP, mu, x, log_floor, omega, r,
                  info_scale, aux0):
    """The write vectors w_t of every token from each variant's gain recursion
    alone (they do not depend on the memory S), and the states the reverse
    sweep needs: the key statistic A_t (PGDN, PKDA), the predicted variance
    p^_t / b^_t (Diagonal / isotropic KDN) with the state before each token."""
    B, T, H, dk = kh.shape
    w = np.zeros_like(kh)
    saved = {}
    if variant in ("gdn", "kda"):
        w = eta[..., None] * kh
    elif variant == "kla":
        w = (eta / (np.sum(kh * kh, axis=-1) + eps))[..., None] * kh
    elif variant in ("pgdn", "pkda"):
        A = np.zeros((B, H, dk)) if aux0 is None else np.array(aux0, dtype=np.float64)
        prev, cur = np.zeros_like(kh), np.zeros_like(kh)
        for t in range(T):
            prev[:, t] = A
            A = alphaP[:, t][..., None] * A + betaP[:, t][..., None] * kh[:, t] ** 2
            cur[:, t] = A
            rr = np.log(np.maximum(A, log_floor)) - mu[None, :, None]
            w[:, t] = eta[:, t][..., None] * np.exp(-np.log(x) * rr / (1 + np.abs(rr))) * kh[:, t]
        saved = dict(prev=prev, cur=cur, final=A)
    elif variant == "kdn":
        p = np.ones((B, H, dk)) if aux0 is None else np.array(aux0, dtype=np.float64)
        prev, cur = np.zeros_like(kh), np.zeros_like(kh)
        for t in range(T):
            prev[:, t] = p
            a = alpha[:, t]
            p_hat = a * a * p + omega[:, t]
            cur[:, t] = p_hat
            kt = kh[:, t]
            w[:, t] = p_hat * kt / (r[:, t] + np.sum(p_hat * kt * kt, axis=-1))[..., None]
            p = p_hat / (1 + (info_scale / r[:, t])[..., None] * kt * kt * p_hat)
        saved = dict(prev=prev, cur=cur, final=p)
    elif variant == "ikdn":
        b = np.ones((B, H)) if aux0 is None else np.array(aux0, dtype=np.float64)
        prev, cur = np.zeros((B, T, H)), np.zeros((B, T, H))
        for t in range(T):
            prev[:, t] = b
            b_hat = np.mean(alpha[:, t] ** 2, axis=-1) * b + omega[:, t]
            cur[:, t] = b_hat
            sk = np.sum(kh[:, t] ** 2, axis=-1)
            w[:, t] = (b_hat / (r[:, t] + b_hat * sk))[..., None] * kh[:, t]
            b = b_hat / (1 + info_scale * sk / (dk * r[:, t]) * b_hat)
        saved = dict(prev=prev, cur=cur, final=b)
    else:
        raise ValueError(f"no gain recursion for variant {variant!r}")
    return w, saved


def _gain_backward(variant, dw, kh, alpha, saved, *, eta, eps, alphaP, betaP, mu, x, log_floor,
                   omega, r, info_scale, daux_T):
    """Reverse sweep of the gain recursion from dL/dw_t (and dL/daux_T): returns
    the key gradient through w, dL/dalpha through the gain (per channel), the
    gate gradients and dL/daux_0."""
    B, T, H, dk = kh.shape
    dk_ = np.zeros_like(kh)
    dal = np.zeros_like(kh)
    g = {}
    if variant in ("gdn", "kda"):
        dk_ = eta[..., None] * dw
        g["deta"] = np.sum(kh * dw, axis=-1)
    elif variant == "kla":
        sk = np.sum(kh * kh, axis=-1) + eps
        kdw = np.sum(kh * dw, axis=-1)
        dk_ = (eta / sk)[..., None] * dw - (2 * eta * kdw / sk ** 2)[..., None] * kh
        g["deta"] = kdw / sk
    elif variant in ("pgdn", "pkda"):
        dA_next = np.zeros((B, H, dk)) if daux_T is None else np.array(daux_T, dtype=np.float64)
        deta, daP, dbP, dmu = (np.zeros((B, T, H)), np.zeros((B, T, H)), np.zeros((B, T, H)),
                               np.zeros(H))
        for t in range(T - 1, -1, -1):
            A, kt = saved["cur"][:, t], kh[:, t]
            rr = np.log(np.maximum(A, log_floor)) - mu[None, :, None]
            Bs = np.exp(-np.log(x) * rr / (1 + np.abs(rr)))
            dk_[:, t] += eta[:, t][..., None] * Bs * dw[:, t]
            deta[:, t] = np.sum(Bs * kt * dw[:, t], axis=-1)
            drr = -np.log(x) * Bs * (eta[:, t][..., None] * kt * dw[:, t]) / (1 + np.abs(rr)) ** 2
            dA = dA_next + np.where(A > log_floor, drr / A, 0.0)
            dmu -= np.sum(np.where(A > log_floor, drr, 0.0), axis=(0, 2))
            daP[:, t] = np.sum(saved["prev"][:, t] * dA, axis=-1)
            dbP[:, t] = np.sum(kt * kt * dA, axis=-1)
            dk_[:, t] += 2 * betaP[:, t][..., None] * kt * dA
            dA_next = alphaP[:, t][..., None] * dA
        g.update(deta=deta, dalphaP=daP, dbetaP=dbP, dmu=dmu, daux0=dA_next)
    elif variant == "kdn":
        dp_next = np.zeros((B, H, dk)) if daux_T is None else np.array(daux_T, dtype=np.float64)
        domega, dr = np.zeros_like(kh), np.zeros((B, T, H))
        for t in range(T - 1, -1, -1):
            p_hat, kt, rt, a = saved["cur"][:, t], kh[:, t], r[:, t], alpha[:, t]
            den = rt + np.sum(p_hat * kt * kt, axis=-1)
            c = np.sum(dw[:, t] * p_hat * kt, axis=-1)
            u = (info_scale / rt)[..., None] * kt * kt
            q1 = 1 + u * p_hat
            dp_hat = dw[:, t] * kt / den[..., None] - (c / den ** 2)[..., None] * kt * kt + dp_next / q1 ** 2
            du = -dp_next * p_hat ** 2 / q1 ** 2
            dk_[:, t] += (dw[:, t] * p_hat / den[..., None] - (2 * c / den ** 2)[..., None] * p_hat * kt
                          + 2 * (info_scale / rt)[..., None] * kt * du)
            dr[:, t] = -c / den ** 2 - info_scale / rt ** 2 * np.sum(kt * kt * du, axis=-1)
            domega[:, t] = dp_hat
            dal[:, t] = 2 * a * saved["prev"][:, t] * dp_hat
            dp_next = a * a * dp_hat
        g.update(domega=domega, dr=dr, daux0=dp_next)
    elif variant == "ikdn":
        db_next = np.zeros((B, H)) if daux_T is None else np.array(daux_T, dtype=np.float64)
        domega, dr = np.zeros((B, T, H)), np.zeros((B, T, H))
        for t in range(T - 1, -1, -1):
            b_hat, kt, rt, a = saved["cur"][:, t], kh[:, t], r[:, t], alpha[:, t]
            sk = np.sum(kt * kt, axis=-1)
            den = rt + b_hat * sk
            uu = info_scale * sk / (dk * rt)
            q1 = 1 + uu * b_hat
            dbeta = np.sum(kt * dw[:, t], axis=-1)
            dk_[:, t] += (b_hat / den)[..., None] * dw[:, t]
            db_hat = dbeta * rt / den ** 2 + db_next / q1 ** 2
            du = -db_next * b_hat ** 2 / q1 ** 2
            dsk = -dbeta * b_hat ** 2 / den ** 2 + du * info_scale / (dk * rt)
            dr[:, t] = -dbeta * b_hat / den ** 2 - du * info_scale * sk / (dk * rt ** 2)
            dk_[:, t] += 2 * dsk[..., None] * kt
            domega[:, t] = db_hat
            dal[:, t] = 2 * a * (saved["prev"][:, t] * db_hat)[..., None] / dk
            db_next = np.mean(a * a, axis=-1) * db_hat
        g.update(domega=domega, dr=dr, daux0=db_next)
    return dk_, dal, g


def chunkwise_backward(q, k, v, log_alpha, variant: str, chunk: int, do, dS_T=None, *,
                       eta=None, eps: float = 1e-6, q_l2norm: bool = False,
                       k_l2norm: bool = False, S0=None, alphaP=None, betaP=None, mu=None,
                       x: float = 1.5, log_floor: float = 1e-12, omega=None, r=None,
                       info_scale: float = 1.0, aux0=None, daux_T=None):
    """The same gradients as ``tokenwise_backward`` (GDN, KLA, KDA) through the
    chunkwise form, chunk by chunk in reverse: the generalised Eqs. (7)-(9) of
    the KLA notes (section 2.5), per chunk with input state S_0,

        R = V - (Gamma.K) S_0,  (I + L) E = R,  O = (Gamma.Q) S_0 + P E,
        S_out = gamma_C . S_0 + Wbar^T E,  Wbar_j = exp(g_C - g_j) . w_j,

    differentiated line by line: dS_0 = gamma_C . dS_out + (Gamma.Q)^T dO
    - (Gamma.K)^T dR;  dE = Wbar dS_out + P^T dO;  dR = (I + L)^-T dE;
    dL = -dR E^T (strictly lower), dP = dO E^T (lower);  dV = dR; and the Gram
    entries L_ij = sum_c k_ic w_jc exp(g_ic - g_jc) (P with q) pass their
    gradients to k, w, q and the log-decay differences.  The per-chunk
    cumulative log-decay g then gives d log alpha_t = sum_{i >= t} dg_i.  The write
    vectors come from each variant's gain recursion, which does not involve the
    memory: the chunk sweep collects dL/dw_t, and a separate reverse gain sweep
    turns it into the gate and gain-state gradients (every chunkwise variant:
    GDN, KLA, KDA, PGDN, PKDA, Diagonal and isotropic KDN).
    """
    if variant not in ("gdn", "kla", "kda", "pgdn", "pkda", "kdn", "ikdn"):
        raise ValueError(f"no chunkwise backward for variant {variant!r}")
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)  # noqa: E731
    q_raw, k_raw, v, la, eta, do = f(q), f(k), f(v), f(log_alpha), f(eta), f(do)
    alphaP, betaP, mu, omega, r = f(alphaP), f(betaP), f(mu), f(omega), f(r)
    B, T, H, dk = k_raw.shape
    dv = v.shape[-1]
    qh = q_raw / np.sqrt(np.sum(q_raw * q_raw, axis=-1, keepdims=True)) if q_l2norm else q_raw
    kh = k_raw / np.sqrt(np.sum(k_raw * k_raw, axis=-1, keepdims=True)) if k_l2norm else k_raw
    per_channel = la.ndim == 4
    gk = dict(eta=eta, eps=eps, alphaP=alphaP, betaP=betaP, mu=mu, x=x, log_floor=log_floor,
              omega=omega, r=r, info_scale=info_scale)
    alpha_c = np.exp(la) if per_channel else np.repeat(np.exp(la)[..., None], dk, axis=-1)
    w_all, gsaved = _gain_forward(variant, kh, alpha_c, aux0=aux0, **gk)
    dw_all = np.zeros_like(kh)
    dq, dk_, dv_ = np.zeros_like(qh), np.zeros_like(kh), np.zeros_like(v)
    dla = np.zeros_like(la)
    dS0_all = np.zeros((B, H, dk, dv))
    starts = list(range(0, T, chunk))
    for b in range(B):
        for h in range(H):
            # forward: the state at every chunk start, and each chunk's pieces
            S = np.zeros((dk, dv)) if S0 is None else f(S0)[b, h].copy()
            saved = []
            for t0 in starts:
                t1 = min(T, t0 + chunk)
                kc, qc, vc = kh[b, t0:t1, h], qh[b, t0:t1, h], v[b, t0:t1, h]
                lac = la[b, t0:t1, h]
                g = np.cumsum(lac, axis=0)
                if not per_channel:
                    g = np.repeat(g[:, None], dk, axis=1)
                wc = w_all[b, t0:t1, h]
                C = t1 - t0
                low_s, low_i = np.tril(np.ones((C, C)), -1), np.tril(np.ones((C, C)), 0)
                ratio = np.exp(g[:, None, :] - g[None, :, :]) * low_i[:, :, None]
                L = np.einsum("ic,jc,ijc->ij", kc, wc, ratio) * low_s
                P = np.einsum("ic,jc,ijc->ij", qc, wc, ratio) * low_i
                Gm = np.exp(g)
                Kg, Qg = kc * Gm, qc * Gm
                A = np.eye(C) + L
                E = np.linalg.solve(A, vc - Kg @ S)
                Wb = np.exp(g[-1][None, :] - g) * wc
                saved.append((t0, t1, kc, qc, wc, g, ratio, L, P, Kg, Qg, A, E, Wb, S.copy()))
                S = np.exp(g[-1])[:, None] * S + Wb.T @ E
            # reverse over chunks
            dS = np.zeros((dk, dv)) if dS_T is None else f(dS_T)[b, h].copy()
            for (t0, t1, kc, qc, wc, g, ratio, L, P, Kg, Qg, A, E, Wb, Sin) in reversed(saved):
                C = t1 - t0
                dOc = do[b, t0:t1, h]
                gC = np.exp(g[-1])
                # S_out = gamma_C . S_in + Wbar^T E
                dSin = gC[:, None] * dS
                dgC = np.sum(dS * Sin, axis=1) * gC                       # d g_C (per channel)
                dWb = E @ dS.T                                            # [C, dk]
                dE = Wb @ dS
                # O = Qg S_in + P E
                dQg = dOc @ Sin.T
                dSin += Qg.T @ dOc
                dP = (dOc @ E.T) * np.tril(np.ones((C, C)), 0)
                dE += P.T @ dOc
                # E = A^-1 R
                dR = np.linalg.solve(A.T, dE)
                dL = -(dR @ E.T) * np.tril(np.ones((C, C)), -1)
                # R = V - Kg S_in
                dv_[b, t0:t1, h] = dR
                dKg = -dR @ Sin.T
                dSin -= Kg.T @ dR
                # Wbar_j = exp(g_C - g_j) . w_j
                eW = np.exp(g[-1][None, :] - g)
                dw = dWb * eW
                dg = np.zeros_like(g)
                dgC = dgC + np.sum(dWb * Wb, axis=0)
                dg -= dWb * Wb
                # L, P entries: X_ijc = a_ic w_jc exp(g_ic - g_jc)
                for Mgrad, Xc, dX in ((dL, kc, "k"), (dP, qc, "q")):
                    X = Xc[:, None, :] * wc[None, :, :] * ratio          # [i, j, c]
                    contrib = Mgrad[:, :, None] * X
                    dg += np.sum(contrib, axis=1)                         # + over j (row i)
                    dg -= np.sum(contrib, axis=0)                         # - over i (column j)
                    dw += np.einsum("ij,ic,ijc->jc", Mgrad, Xc, ratio)
                    da = np.einsum("ij,jc,ijc->ic", Mgrad, wc, ratio)
                    if dX == "k":
                        dk_[b, t0:t1, h] += da
                    else:
                        dq[b, t0:t1, h] += da
                # Kg = k . exp(g), Qg = q . exp(g)
                Gm = np.exp(g)
                dk_[b, t0:t1, h] += dKg * Gm
                dq[b, t0:t1, h] += dQg * Gm
                dg += dKg * Kg + dQg * Qg
                dg[-1] += dgC
                dw_all[b, t0:t1, h] = dw
                # g = cumsum(log alpha): reverse cumulative sum (scalar decay: over channels too)
                rc = np.cumsum(dg[::-1], axis=0)[::-1]
                dla[b, t0:t1, h] = rc if per_channel else np.sum(rc, axis=1)
                dS = dSin
            dS0_all[b, h] = dS
    # the gain recursion's reverse sweep from dL/dw
    dk_g, dal_g, gg = _gain_backward(variant, dw_all, kh, alpha_c, gsaved, daux_T=f(daux_T), **gk)
    dk_ += dk_g
    if per_channel:
        dla += alpha_c * dal_g
    elif variant not in ("gdn", "kla", "pgdn"):
        raise ValueError("a per-channel gain needs per-channel decay")
    if q_l2norm:
        dq = _norm_backward(q_raw, dq)
    if k_l2norm:
        dk_ = _norm_backward(k_raw, dk_)
    out = dict(dq=dq, dk=dk_, dv=dv_, dlog_alpha=dla, dS0=dS0_all)
    out.update(gg)
    return out
