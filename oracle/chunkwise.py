"""Naive chunkwise fp64 oracle: the chunk-parallel restatement, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Within a chunk of C tokens with input state S_0, let g_i be the cumulative
log-decay from the chunk start to token i (a scalar, or a dk-vector for
per-channel decay), so gamma_i = exp(g_i) and the ratio gamma_i/gamma_j is
formed as exp(g_i - g_j) (KDN notes section 6, numerics paragraph).  Writing
E for the per-token residuals e_i and W for the rows w_j, unrolling the
recurrence gives the generalisation of KLA notes Eqs. (7)-(9) (section 2.5)
to an arbitrary write matrix W (and of the PDN two-key form, section 2.6):

    L_ij = sum_c k_ic w_jc exp(g_ic - g_jc)          j <  i   (strict lower)
    P_ij = sum_c q_ic w_jc exp(g_ic - g_jc)          j <= i   (diagonal kept)
    (I + L) E = V - (Gamma . K) S_0                                   (7)
    O = (Gamma . Q) S_0 + P E                                         (8)
    S_out = diag(gamma_C) S_0 + sum_j (exp(g_C - g_j) . w_j) e_j^T    (9)

With W = diag(beta) K and scalar decay, U = diag(beta) E is exactly the U of
Eq. (7).  The unit lower-triangular system is solved by plain forward
substitution.  Ratios use gamma_i/gamma_j (a write decays only after it is
made), the reading the KLA notes (appendix-notation paragraph of section 2.5)
confirm yields Eqs. (7)-(9).

The write vectors are produced chunk by chunk with the pages' chunked gain
forms rather than token by token:
  * PGDN statistic: A_out = (prod alphaP) A_in + sum_j (prod_{l>j} alphaP_l)
    betaP_j k_j^2 (PDN notes section 2.6, last paragraph), evaluated for every
    prefix of the chunk;
  * KDN variance: products of the 2x2 Moebius matrices
    M_t = [[alpha^2, omega], [u alpha^2, 1 + u omega]] acting on the
    homogeneous pair (n, d) with p = n/d (KDN notes section 6, Eqs. (32)-(39));
    the isotropic variance b is the same scan with one channel, the mean
    squared decay in place of alpha^2 (KDN notes section 7: "this scalar
    recursion can also be written as a 2x2 Moebius scan").
"""

from __future__ import annotations

import numpy as np

from .recurrence import VARIANTS, l2normalize, pgdn_squash


def pgdn_stat_chunk(A_in, k2, log_alphaP, betaP):
    """Statistic A_t at every token of one chunk from the chunk-entry A_in.

    A_in [dk]; k2 [C, dk] = k*k; log_alphaP, betaP [C].
    A_t = exp(a_t) A_in + sum_{j<=t} exp(a_t - a_j) betaP_j k2_j with a the
    cumulative sum of log alphaP (the closed form of the decayed linear scan).
    """
    a = np.cumsum(log_alphaP)
    C = k2.shape[0]
    out = np.empty_like(k2)
    for t in range(C):
        wts = np.exp(a[t] - a[: t + 1]) * betaP[: t + 1]
        out[t] = np.exp(a[t]) * A_in + wts @ k2[: t + 1]
    return out


def kdn_mobius_chunk(p_in, alpha, omega, u):
    """Variances p_{t-1} (prior of token t) and p_t for one chunk via Moebius products.

    p_in [dk]; alpha, omega, u [C, dk].  For each channel the scaled variance
    recurrence is the fractional-linear map p -> (a p + b)/(c p + d) with
    matrix M_t = [[alpha^2, omega], [u alpha^2, 1 + u omega]].  The prefix
    product M_t ... M_1 applied to (p_in, 1) gives (n_t, d_t), p_t = n_t/d_t.
    Returns (p_prev [C, dk], p_post [C, dk]).
    """
    C, dk = alpha.shape
    a2 = alpha * alpha
    # prefix products, one 2x2 matrix per channel: Pm[c] = M_t ... M_1
    Pm = np.broadcast_to(np.eye(2), (dk, 2, 2)).copy()
    p_prev = np.empty((C, dk))
    p_post = np.empty((C, dk))
    for t in range(C):
        n0 = Pm[:, 0, 0] * p_in + Pm[:, 0, 1]
        d0 = Pm[:, 1, 0] * p_in + Pm[:, 1, 1]
        p_prev[t] = n0 / d0
        Mt = np.empty((dk, 2, 2))
        Mt[:, 0, 0] = a2[t]
        Mt[:, 0, 1] = omega[t]
        Mt[:, 1, 0] = u[t] * a2[t]
        Mt[:, 1, 1] = 1.0 + u[t] * omega[t]
        Pm = Mt @ Pm
        p_post[t] = (Pm[:, 0, 0] * p_in + Pm[:, 0, 1]) / (Pm[:, 1, 0] * p_in + Pm[:, 1, 1])
    return p_prev, p_post


def _chunk_solve(q, k, v, w, g, S0):
    """Eqs. (7)-(9) generalised, for one (batch, head) and one chunk.

    q, k, w [C, dk]; v [C, dv]; g [C, dk] cumulative log-decay (a scalar
    decay is broadcast over dk); S0 [dk, dv].  Returns (O [C, dv], S_out).
    """
    C = k.shape[0]
    ratio = np.exp(g[:, None, :] - g[None, :, :])            # [i, j, c] = exp(g_ic - g_jc)
    lower_strict = np.tril(np.ones((C, C)), -1)
    lower_incl = np.tril(np.ones((C, C)), 0)
    # only j <= i entries are used; masked entries may be exp(positive), zero them first
    ratio = ratio * lower_incl[:, :, None]
    L = np.einsum("ic,jc,ijc->ij", k, w, ratio) * lower_strict
    P = np.einsum("ic,jc,ijc->ij", q, w, ratio) * lower_incl
    gamma = np.exp(g)                                          # [C, dk]
    rhs = v - (gamma * k) @ S0
    E = np.empty_like(rhs)
    for i in range(C):                                         # forward substitution, unit diagonal
        E[i] = rhs[i] - L[i, :i] @ E[:i]
    O = (gamma * q) @ S0 + P @ E
    S_out = np.exp(g[-1])[:, None] * S0 + (np.exp(g[-1][None, :] - g) * w).T @ E
    return O, S_out


def chunkwise(q, k, v, log_alpha, variant: str, chunk: int, *, eta=None,
              eps: float = 1e-6, q_l2norm: bool = False, k_l2norm: bool = False,
              alphaP=None, betaP=None, mu=None, x: float = 1.5,
              log_floor: float = 1e-12, omega=None, r=None,
              info_scale: float = 1.0, S0=None, aux0=None):
    """Chunkwise forward over [B, T, H, d] inputs, same arguments as ``tokenwise``.

    T need not be a multiple of ``chunk``: the last chunk is shorter.
    Returns (o, S_T, aux_T) like ``tokenwise``.
    """
    if variant not in VARIANTS:
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
    per_channel = log_alpha.ndim == 4

    o = np.zeros((B, T, H, dv))
    S_fin = np.zeros((B, H, dk, dv))
    aux_fin = (None if variant in ("gdn", "kla", "kda")
               else np.zeros((B, H)) if variant == "ikdn" else np.zeros((B, H, dk)))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], dtype=np.float64)
            if variant in ("pgdn", "pkda"):
                aux = np.zeros(dk) if aux0 is None else np.array(aux0[b, h], dtype=np.float64)
            elif variant == "kdn":
                aux = np.ones(dk) if aux0 is None else np.array(aux0[b, h], dtype=np.float64)
            elif variant == "ikdn":
                aux = 1.0 if aux0 is None else float(aux0[b, h])
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                kc, qc, vc = k[b, t0:t1, h], q[b, t0:t1, h], v[b, t0:t1, h]
                la = log_alpha[b, t0:t1, h]
                g = np.cumsum(la, axis=0)
                if not per_channel:
                    g = np.repeat(g[:, None], dk, axis=1)
                if variant in ("gdn", "kda"):
                    w = eta[b, t0:t1, h][:, None] * kc
                elif variant == "kla":
                    w = (eta[b, t0:t1, h] / (np.sum(kc * kc, axis=1) + eps))[:, None] * kc
                elif variant in ("pgdn", "pkda"):
                    A = pgdn_stat_chunk(aux, kc * kc, np.log(alphaP[b, t0:t1, h]), betaP[b, t0:t1, h])
                    aux = A[-1]
                    w = eta[b, t0:t1, h][:, None] * pgdn_squash(A, mu[h], x, log_floor) * kc
                elif variant == "ikdn":
                    rc = r[b, t0:t1, h]
                    kk = np.sum(kc * kc, axis=1)
                    a_mean = np.mean(np.exp(2.0 * la), axis=1)          # [C]
                    u = info_scale * kk / (dk * rc)
                    om = omega[b, t0:t1, h]
                    b_prev, b_post = kdn_mobius_chunk(np.array([aux]), np.sqrt(a_mean)[:, None],
                                                      om[:, None], u[:, None])
                    aux = float(b_post[-1, 0])
                    b_hat = a_mean * b_prev[:, 0] + om
                    w = (b_hat / (rc + b_hat * kk))[:, None] * kc
                else:
                    rc = r[b, t0:t1, h]
                    u = (info_scale / rc)[:, None] * kc * kc
                    alpha = np.exp(la)
                    p_prev, p_post = kdn_mobius_chunk(aux, alpha, omega[b, t0:t1, h], u)
                    aux = p_post[-1]
                    p_hat = alpha * alpha * p_prev + omega[b, t0:t1, h]
                    w = p_hat * kc / (rc + np.sum(p_hat * kc * kc, axis=1))[:, None]
                O, S = _chunk_solve(qc, kc, vc, w, g, S)
                o[b, t0:t1, h] = O
            S_fin[b, h] = S
            if aux_fin is not None:
                aux_fin[b, h] = aux
    return o, S_fin, aux_fin
