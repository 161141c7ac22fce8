"""Tokenwise fp64 oracle: the plain definition of the recurrence.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the product
imports this module.

The unified recurrence (Kalman Delta Networks notes, section 1 "From storing
every token to storing a map", the displayed equation and the table under it):

    S~_t = D_t S_{t-1}
    e_t  = v_t - S~_t^T k_t
    S_t  = S~_t + w_t e_t^T
    o_t  = S_t^T q_t                    (read after the write)

with S in R^{dk x dv}, D_t = alpha_t I (GDN, KLA, PGDN) or diag(alpha_t)
(KDA, PKDA, Diagonal KDN), and a per-variant write vector w_t:

    GDN   w = eta k                                 (KLA notes section 1.1)
    KDA   w = eta k, D_t = diag(alpha_t)            (KDN notes section 1, table)
    KLA   w = eta k / (||k||^2 + eps)               (KLA notes Eq. (3), Alg. 1)
    PGDN  A_t = alphaP A_{t-1} + betaP (k*k)        (PDN notes Eq. (9))
          r = log max(A_t, floor) - mu ; s = r / (1 + |r|)
          B = exp(-log(x) s) ;  w = beta (B * k)
    PKDA  the PGDN write key with D_t = diag(alpha_t)   (PDN notes section 2.5)
    IKDN  isotropic KDN, one variance b per head       (KDN notes section 7, Eq. (40))
          a = mean_i alpha_i^2 ; b^ = a b_{t-1} + omega ; beta = b^ / (r + b^ ||k||^2)
          w = beta k ; b_t = b^ / (1 + u b^), u = mu ||k||^2 / (dk r)
    EKDN  exact Kalman memory, dense key covariance P   (KDN notes section 2.2,
          P^ = D P D^T + diag(omega) ; w = P^ k / (r + k^T P^ k)   Eqs. (12)-(17))
          P_t = (I - w k^T) P^       (tokenwise only: the pages give it no chunk form)
    KDN   p^ = alpha^2 * p_{t-1} + omega            (KDN notes Eq. (23))
          kappa = p^ * k / (r + sum(p^ k^2)) ; w = kappa
          p_t = p^ / (1 + (mu/r) k*k * p^)          (KDN notes Eqs. (60)-(65))

Layouts follow the library: tokens are [B, T, H, d]; per-token scalars are
[B, T, H]; per-channel gates (KDA, PKDA and KDN log-alpha, KDN omega) are
[B, T, H, dk]; the
state is [B, H, dk, dv].  Everything is computed in float64.
"""

from __future__ import annotations

import numpy as np

VARIANTS = ("gdn", "kla", "pgdn", "kdn", "kda", "pkda", "ikdn")
TOKENWISE_ONLY = ("ekdn",)   # a dense Riccati recursion, no chunkwise restatement


def l2normalize(x: np.ndarray, floor: float = 1e-30) -> np.ndarray:
    """x / max(||x||_2, floor) along the last axis.

    Query normalisation at readout is KLA notes Eq. (3) (o = S^T q/||q||);
    key normalisation is the L2-normalised q/k of the PDN architecture (PDN
    notes section 3.1, table "training and architecture").
    """
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, floor)


# ---------------------------------------------------------------- write vectors

def gdn_write(k: np.ndarray, eta: np.ndarray) -> np.ndarray:
    """GDN write vector w = beta k with beta = eta (KLA notes section 1.1)."""
    return eta[..., None] * k


def kla_write(k: np.ndarray, eta: np.ndarray, eps: float) -> np.ndarray:
    """Kaczmarz write vector w = eta/(||k||^2 + eps) k (KLA notes Eq. (3))."""
    energy = np.sum(k * k, axis=-1)
    return (eta / (energy + eps))[..., None] * k


def pgdn_stat_update(A_prev, k, alphaP, betaP):
    """Decayed diagonal key statistic A_t = alphaP A_{t-1} + betaP (k*k).

    PDN notes section 2.4, Eq. (9) (first line).  alphaP, betaP are scalars
    per (batch, head); A is a dk-vector per (batch, head).
    """
    return alphaP[..., None] * A_prev + betaP[..., None] * (k * k)


def pgdn_squash(A, mu, x: float, floor: float):
    """Bounded write-key scale B = exp(-log(x) * r/(1+|r|)), r = log A - mu.

    PDN notes section 2.4, Eq. (9) (second and third lines).  The log guard
    ``log max(A, floor)`` is the reading for the unspecified guard the notes
    flag in the same section.  ``mu`` broadcasts against A's leading axes.
    """
    r = np.log(np.maximum(A, floor)) - mu
    s = r / (1.0 + np.abs(r))
    return np.exp(-np.log(x) * s)


def kdn_predict(p_prev, alpha, omega):
    """Predicted diagonal variance p^ = alpha^2 * p + omega (KDN notes Eq. (23))."""
    return alpha * alpha * p_prev + omega


def kdn_gain(p_hat, k, r):
    """Diagonal Kalman gain kappa = p^ k / (r + sum_i p^_i k_i^2) (KDN Eq. (23))."""
    z = np.sum(p_hat * k * k, axis=-1)
    return p_hat * k / (r + z)[..., None]


def kdn_variance_update(p_hat, k, r, mu: float):
    """Reverse-KL diagonal variance with information scaling mu.

    p = p^ / (1 + u p^), u = (mu / r) k*k  (KDN notes section 5, Eqs. (60)-(65));
    mu = 1 is the strict reverse-KL projection p_i = (1/p^_i + k_i^2/r)^-1.
    """
    u = (mu / r)[..., None] * (k * k)
    return p_hat / (1.0 + u * p_hat)


def ikdn_predict(b_prev, alpha, omega):
    """Isotropic predicted variance b^ = a b + omega, a = (1/dk) sum_i alpha_i^2.

    The prediction keeps P = b I by projecting D P D onto multiples of I by its
    trace, i.e. the mean eigenvalue (KDN notes section 7, Eq. (40)); alpha may
    still differ per channel.  b_prev, omega [...]; alpha [..., dk].
    """
    return np.mean(alpha * alpha, axis=-1) * b_prev + omega


def ikdn_gain(b_hat, k, r):
    """Isotropic gain: w = beta k, beta = b^ / (r + b^ ||k||^2) (KDN Eq. (40))."""
    beta = b_hat / (r + b_hat * np.sum(k * k, axis=-1))
    return beta[..., None] * k


def ikdn_variance_update(b_hat, k, r, mu: float):
    """Reverse-KL isotropic variance with information scaling mu (KDN Eq. (40)):
    b = b^ / (1 + u b^), u = mu ||k||^2 / (dk r) (the harmonic mean of the
    posterior eigenvalues)."""
    u = mu * np.sum(k * k, axis=-1) / (k.shape[-1] * r)
    return b_hat / (1.0 + u * b_hat)


def ekdn_predict(P_prev, alpha, omega):
    """Predicted dense key covariance P^ = D P D^T + diag(omega), D = diag(alpha)
    (KDN notes section 2.2, Eq. (12)).  P [..., dk, dk]; alpha, omega [..., dk]."""
    P_hat = alpha[..., :, None] * P_prev * alpha[..., None, :]
    return P_hat + omega[..., :, None] * np.eye(P_prev.shape[-1])


def ekdn_gain(P_hat, k, r):
    """Kalman gain kappa = P^ k / (r + k^T P^ k) (KDN notes section 2.2, Eq. (13))."""
    Pk = np.einsum("...ij,...j->...i", P_hat, k)
    return Pk / (r + np.sum(k * Pk, axis=-1))[..., None]


def ekdn_cov_update(P_hat, kappa, k):
    """Posterior covariance P = (I - kappa k^T) P^ (KDN notes section 2.2, Eq. (15))."""
    return P_hat - kappa[..., :, None] * np.einsum("...j,...jl->...l", k, P_hat)[..., None, :]


# ---------------------------------------------------------------- the recurrence

def recurrence_step(S, q, k, v, decay, w):
    """One token of the unified recurrence, for every (batch, head) at once.

    S [..., dk, dv]; q, k, w [..., dk]; v [..., dv]; decay is alpha, either a
    scalar per head ([...]) or a dk-vector per head ([..., dk]) that scales
    the rows of S (D_t = diag(alpha_t)).  Returns (S_t, o_t, e_t).
    """
    if decay.ndim == S.ndim - 2:           # scalar decay
        S_tilde = decay[..., None, None] * S
    else:                                   # per-channel decay: rows of S
        S_tilde = decay[..., :, None] * S
    e = v - np.einsum("...kv,...k->...v", S_tilde, k)
    S_new = S_tilde + w[..., :, None] * e[..., None, :]
    o = np.einsum("...kv,...k->...v", S_new, q)
    return S_new, o, e


def tokenwise(q, k, v, log_alpha, variant: str, *, eta=None, eps: float = 1e-6,
              q_l2norm: bool = False, k_l2norm: bool = False,
              alphaP=None, betaP=None, mu=None, x: float = 1.5,
              log_floor: float = 1e-12, omega=None, r=None,
              info_scale: float = 1.0, S0=None, aux0=None, return_trace=False):
    """Run the recurrence token by token over [B, T, H, d] inputs in float64.

    variant  one of VARIANTS.
    eta      [B,T,H]: GDN/KLA eta, PGDN beta.
    alphaP, betaP [B,T,H]; mu [H]          PGDN / PKDA statistic gates and centre.
    omega [B,T,H,dk]; r [B,T,H]            KDN process / observation noise
                                           (isotropic KDN: omega [B,T,H]).
    log_alpha [B,T,H] (scalar decay) or [B,T,H,dk] (KDA, PKDA, KDN).
    S0 [B,H,dk,dv] (None = 0); aux0 [B,H,dk]: PGDN / PKDA A_0 (None = 0) or
    KDN p_0 (None = 1); isotropic KDN b_0 [B,H] (None = 1); exact Kalman P_0
    [B,H,dk,dk] (None = I).
    Returns (o [B,T,H,dv], S_T [B,H,dk,dv], aux_T [B,H,dk] or None); with
    ``return_trace`` also a dict of per-token write vectors and residuals.
    """
    if variant not in VARIANTS + TOKENWISE_ONLY:
        raise ValueError(f"unknown variant {variant!r}")
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)  # noqa: E731
    q, k, v, log_alpha = f(q), f(k), f(v), f(log_alpha)
    eta, alphaP, betaP, mu, omega, r = f(eta), f(alphaP), f(betaP), f(mu), f(omega), f(r)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if q_l2norm:
        q = l2normalize(q)
    if k_l2norm:
        k = l2normalize(k)

    S = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    aux = None
    if variant in ("pgdn", "pkda"):
        aux = np.zeros((B, H, dk)) if aux0 is None else np.array(aux0, dtype=np.float64)
    elif variant == "kdn":
        aux = np.ones((B, H, dk)) if aux0 is None else np.array(aux0, dtype=np.float64)
    elif variant == "ikdn":
        aux = np.ones((B, H)) if aux0 is None else np.array(aux0, dtype=np.float64)
    elif variant == "ekdn":   # dense covariance P [B, H, dk, dk], P_0 = I by default
        aux = (np.broadcast_to(np.eye(dk), (B, H, dk, dk)).copy() if aux0 is None
               else np.array(aux0, dtype=np.float64))

    o = np.zeros((B, T, H, dv))
    trace = {"w": np.zeros((B, T, H, dk)), "e": np.zeros((B, T, H, dv))} if return_trace else None
    for t in range(T):
        kt, qt, vt = k[:, t], q[:, t], v[:, t]
        alpha = np.exp(log_alpha[:, t])
        if variant in ("gdn", "kda"):
            w = gdn_write(kt, eta[:, t])
        elif variant == "kla":
            w = kla_write(kt, eta[:, t], eps)
        elif variant in ("pgdn", "pkda"):
            aux = pgdn_stat_update(aux, kt, alphaP[:, t], betaP[:, t])
            Bscale = pgdn_squash(aux, mu[None, :, None], x, log_floor)
            w = eta[:, t][..., None] * (Bscale * kt)
        elif variant == "ekdn":
            P_hat = ekdn_predict(aux, alpha, omega[:, t])
            w = ekdn_gain(P_hat, kt, r[:, t])
            aux = ekdn_cov_update(P_hat, w, kt)
        elif variant == "ikdn":
            b_hat = ikdn_predict(aux, alpha, omega[:, t])
            w = ikdn_gain(b_hat, kt, r[:, t])
            aux = ikdn_variance_update(b_hat, kt, r[:, t], info_scale)
        else:  # kdn: predict, gain, (memory update below), variance update
            p_hat = kdn_predict(aux, alpha, omega[:, t])
            w = kdn_gain(p_hat, kt, r[:, t])
            aux = kdn_variance_update(p_hat, kt, r[:, t], info_scale)
        S, o[:, t], e = recurrence_step(S, qt, kt, vt, alpha, w)
        if return_trace:
            trace["w"][:, t], trace["e"][:, t] = w, e
    if return_trace:
        return o, S, aux, trace
    return o, S, aux
