"""Side oracles fixed by closed forms (fp64, CPU).  TEST INFRASTRUCTURE ONLY.

These are not part of the hot path; they pin the recurrence oracle from
outside.  State orientation follows the rest of the oracle: S is dk x dv and
o = S^T q (the PDN notes write the transpose, S in R^{dv x dk} with o = S q;
every formula here is that one transposed).

* Exact ridge test-time regression (PDN notes section 2.1, Eqs. (1)-(2)):
  G_t = lam I + sum k k^T, C_t = sum k v^T, S*_t = G_t^{-1} C_t.
* ATK: the same solution as a delta rule with read key k and write key
  k~_t = P_{t-1} k_t / (1 + k_t^T P_{t-1} k_t), P = G^{-1} tracked by
  Sherman-Morrison (PDN notes section 2.2, Theorem 3.1, Eqs. (3)-(5)).
* The diagonal approximation and its counterexample (PDN notes section 2.3).
* A dense-covariance Kalman filter (KDN notes section 2, Eqs. (12)-(17)),
  to which Diagonal KDN reduces when the keys keep the covariance diagonal.
"""

from __future__ import annotations

import numpy as np


def ridge_atq(q, k, v, lam: float):
    """Exact ridge readout o_t = (S*_t)^T q_t with S*_t = G_t^{-1} C_t.

    q, k [T, dk]; v [T, dv].  Solved with a dense linear solve per token.
    Returns (o [T, dv], S*_T [dk, dv]).
    """
    T, dk = k.shape
    G = lam * np.eye(dk)
    C = np.zeros((dk, v.shape[1]))
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        G += np.outer(k[t], k[t])
        C += np.outer(k[t], v[t])
        S = np.linalg.solve(G, C)
        o[t] = S.T @ q[t]
    return o, S


def atk_write_keys(k, lam: float):
    """Write keys k~_t of the exact ATK recursion (Sherman-Morrison on P = G^{-1}).

    k [T, dk].  P_0 = I / lam;  k~_t = P_{t-1} k_t / (1 + k_t^T P_{t-1} k_t);
    P_t = P_{t-1} - P_{t-1} k_t k_t^T P_{t-1} / (1 + k_t^T P_{t-1} k_t).
    """
    T, dk = k.shape
    P = np.eye(dk) / lam
    out = np.zeros_like(k, dtype=np.float64)
    for t in range(T):
        Pk = P @ k[t]
        denom = 1.0 + k[t] @ Pk
        out[t] = Pk / denom
        P = P - np.outer(Pk, Pk) / denom
    return out


def diagonal_atq_state(k, v, lam: float):
    """State of the diagonal ATQ readout: diag(lam + sum k*k)^{-1} sum k v^T."""
    A = lam + np.sum(k * k, axis=0)
    return (k.T @ v) / A[:, None]


def diagonal_atk_write_keys(k, lam: float):
    """Write keys when P_{t-1} is replaced by the diagonal inverse diag(A_{t-1})^{-1}."""
    T, dk = k.shape
    A = np.full(dk, lam, dtype=np.float64)
    out = np.zeros_like(k, dtype=np.float64)
    for t in range(T):
        Pk = k[t] / A
        out[t] = Pk / (1.0 + k[t] @ Pk)
        A = A + k[t] * k[t]
    return out


def dense_kalman(q, k, v, alpha, omega, r, P0):
    """Exact Kalman memory with dense key-space covariance, D = diag(alpha), Omega = diag(omega).

    q, k [T, dk]; v [T, dv]; alpha, omega [T, dk]; r [T]; P0 [dk, dk].
    Predict S^ = D S, P^ = D P D^T + Omega; gain kappa = P^ k/(r + k^T P^ k);
    S = S^ + kappa (v - S^T k)^T; P = (I - kappa k^T) P^; o = S^T q.
    Returns (o [T, dv], S_T, P_T, kappas [T, dk]).
    """
    T, dk = k.shape
    S = np.zeros((dk, v.shape[1]))
    P = np.array(P0, dtype=np.float64)
    o = np.zeros((T, v.shape[1]))
    kappas = np.zeros((T, dk))
    for t in range(T):
        D = np.diag(alpha[t])
        S_hat = D @ S
        P_hat = D @ P @ D.T + np.diag(omega[t])
        Pk = P_hat @ k[t]
        kappa = Pk / (r[t] + k[t] @ Pk)
        S = S_hat + np.outer(kappa, v[t] - S_hat.T @ k[t])
        P = (np.eye(dk) - np.outer(kappa, k[t])) @ P_hat
        o[t] = S.T @ q[t]
        kappas[t] = kappa
    return o, S, P, kappas
