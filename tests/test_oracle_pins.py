"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (fixtures under tests/golden/, each with its citation), a closed
form, a library routine (dense solve, least squares, eigenvalues), a
special case that reduces to another method, or brute-force agreement of
two independently written forms (tokenwise vs chunkwise).
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ridge

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


def one_token(k, v, eta, variant="kla", eps=0.0, log_alpha=0.0):
    """Run the tokenwise oracle on a single 1-d token with read key = k."""
    arr = lambda x: np.array(x, dtype=np.float64).reshape(1, 1, 1, -1)  # noqa: E731
    sc = lambda x: np.array(x, dtype=np.float64).reshape(1, 1, 1)  # noqa: E731
    o, S, _ = oracle.tokenwise(arr(k), arr(k), arr(v), sc(log_alpha), variant, eta=sc(eta), eps=eps)
    return S[0, 0, 0, 0], o[0, 0, 0, 0]


# ------------------------------------------------------------------ P1: KLA worked example

def test_kla_worked_example():
    g = golden("kla_worked_example.json")
    # plain delta rule with beta = 1 (GDN with eta = 1, no decay)
    S, read = one_token(2.0, 1.0, 1.0, variant="gdn")
    assert S == pytest.approx(g["delta_rule_beta_1"]["S"], abs=1e-15)
    assert read == pytest.approx(g["delta_rule_beta_1"]["read"], abs=1e-15)
    assert 1.0 - read == pytest.approx(g["delta_rule_beta_1"]["residual_after"], abs=1e-15)
    # Kaczmarz step, eta = 1, eps = 0: the constraint holds exactly
    S, read = one_token(2.0, 1.0, 1.0, variant="kla", eps=0.0)
    assert S == pytest.approx(g["kla_eta_1_eps_0"]["S"], abs=1e-15)
    assert read == pytest.approx(g["kla_eta_1_eps_0"]["read"], abs=1e-15)
    # eta = 1/2 corrects half of the residual
    S, read = one_token(2.0, 1.0, 0.5, variant="kla", eps=0.0)
    assert S == pytest.approx(g["kla_eta_half_eps_0"]["S"], abs=1e-15)
    assert 1.0 - read == pytest.approx(g["kla_eta_half_eps_0"]["residual_after"], abs=1e-15)
    # with the stabiliser eps = 1e-6 the read is 4/(4+eps)
    e = g["kla_eta_1_eps_1e-6"]
    S, read = one_token(2.0, 1.0, 1.0, variant="kla", eps=e["eps"])
    assert read == pytest.approx(e["read"], abs=5e-9)


# ------------------------------------------------------------------ shared random inputs

def random_inputs(variant, B=2, T=37, H=2, dk=8, dv=6, seed=0, decay_shift=0.5):
    """Inputs with the workloads' distributions at tiny sizes (float64)."""
    r = rng(seed)
    d = dict(q=r.standard_normal((B, T, H, dk)), k=r.standard_normal((B, T, H, dk)),
             v=r.standard_normal((B, T, H, dv)))
    sig = lambda x: 1 / (1 + np.exp(-x))  # noqa: E731
    sp = lambda x: np.log1p(np.exp(x))  # noqa: E731
    if variant in ("gdn", "kla", "pgdn", "kda", "pkda"):
        d["eta"] = sig(r.standard_normal((B, T, H)))
        d["log_alpha"] = -sp(r.standard_normal((B, T, H)) + decay_shift)
    if variant in ("pgdn", "pkda"):
        d["alphaP"] = sig(r.standard_normal((B, T, H)) + 3)
        d["betaP"] = sig(r.standard_normal((B, T, H)))
        d["mu"] = np.exp(0.5 * r.standard_normal(H))
    if variant in ("kda", "pkda"):   # per-channel decay
        d["log_alpha"] = -sp(r.standard_normal((B, T, H, dk)) + decay_shift)
    if variant == "kdn":
        d["log_alpha"] = -sp(r.standard_normal((B, T, H, dk)) + decay_shift)
        d["omega"] = sp(r.standard_normal((B, T, H, dk)) - 3)
        d["r"] = sp(r.standard_normal((B, T, H)))
    if variant == "ikdn":   # one process noise per (b, t, h)
        d["log_alpha"] = -sp(r.standard_normal((B, T, H, dk)) + decay_shift)
        d["omega"] = sp(r.standard_normal((B, T, H)) - 3)
        d["r"] = sp(r.standard_normal((B, T, H)))
    return d


def call(fn, variant, d, **kw):
    args = {k: d[k] for k in ("eta", "alphaP", "betaP", "mu", "omega", "r") if k in d}
    args.update(kw)
    return fn(d["q"], d["k"], d["v"], d["log_alpha"], variant, **args)


# ------------------------------------------------------------------ P2: residual contraction

@pytest.mark.parametrize("variant", oracle.VARIANTS)
def test_residual_contraction_every_step(variant):
    """Re-reading with k after the write leaves e+ = (1 - k^T w) e (KLA notes Eq. (5))."""
    d = random_inputs(variant, seed=1)
    o, S, aux, tr = call(oracle.tokenwise, variant, d, return_trace=True, eps=1e-6)
    # rerun step by step to re-read each post-write state with the same key
    B, T, H, dk = d["k"].shape
    S_t = np.zeros((B, H, dk, d["v"].shape[-1]))
    for t in range(T):
        alpha = np.exp(d["log_alpha"][:, t])
        w = tr["w"][:, t]
        S_t, _, e = oracle.recurrence_step(S_t, d["q"][:, t], d["k"][:, t], d["v"][:, t], alpha, w)
        e_plus = d["v"][:, t] - np.einsum("bhkv,bhk->bhv", S_t, d["k"][:, t])
        factor = 1.0 - np.sum(d["k"][:, t] * w, axis=-1)
        np.testing.assert_allclose(e_plus, factor[..., None] * e, rtol=1e-9, atol=1e-12)
        if variant == "kla":   # factor = 1 - eta ||k||^2/(||k||^2+eps) in [0, 1)
            assert np.all(factor >= 0) and np.all(factor < 1)
        if variant == "kdn":   # factor = r/(r+z): beta_eff = z/(r+z) in [0, 1)
            assert np.all(factor > 0) and np.all(factor <= 1)


# ------------------------------------------------------------------ P3: PDN squash

def test_pdn_squash_example():
    g = golden("pdn_squash_example.json")
    B = oracle.pgdn_squash(np.array(g["A"]), math.log(4.0), g["x"], 1e-12)
    tol = 0.5 * 10 ** -g["printed_decimals"]
    np.testing.assert_allclose(B, g["B_printed"], atol=tol)
    # r = +-ln 4 gives s = +-ln4/(1+ln4) and B = x^(-s): the two entries are reciprocal
    assert B[0] * B[1] == pytest.approx(1.0, abs=1e-14)


def test_pdn_write_key_inner_product_bounds():
    """k^T k~ in [1/x, x] for unit k (PDN notes section 2.7, App. E.3)."""
    r = rng(3)
    x = 1.5
    A = np.exp(6 * r.standard_normal((1000, 16)))
    k = oracle.l2normalize(r.standard_normal((1000, 16)))
    B = oracle.pgdn_squash(A, 0.3, x, 1e-12)
    ip = np.sum(k * B * k, axis=-1)
    assert np.all(B > 1 / x) and np.all(B < x)
    assert np.all(ip >= 1 / x) and np.all(ip <= x)


def test_pgdn_step_spectrum():
    """The PGDN transition alpha (I - beta k k~^T) has eigenvalues alpha (x dk-1)
    and alpha (1 - beta k^T k~) (PDN notes section 2.7, App. E.3).  The transition
    is read off the oracle's own step with v = 0 applied to S = I."""
    r = rng(4)
    dk = 6
    k = oracle.l2normalize(r.standard_normal(dk))
    kt = oracle.pgdn_squash(np.exp(r.standard_normal(dk)), 0.2, 1.5, 1e-12) * k
    alpha, beta = 0.8, 0.7
    w = beta * kt
    S1, _, _ = oracle.recurrence_step(np.eye(dk), k, k, np.zeros(dk), np.array(alpha), w)
    ev = np.sort(np.linalg.eigvals(S1.T).real)  # S_t = M S with M the transition; S1 = M
    expect = np.sort(np.r_[np.full(dk - 1, alpha), alpha * (1 - beta * k @ kt)])
    np.testing.assert_allclose(ev, expect, atol=1e-12)


# ------------------------------------------------------------------ P4: ridge regression ATQ = ATK

def test_exact_atq_equals_atk_delta_rule():
    """The generic recurrence core with exact ATK write keys (D = I) reproduces the
    dense ridge solution at every token (PDN notes Theorem 3.1, Eqs. (3)-(5))."""
    r = rng(5)
    T, dk, dv, lam = 40, 5, 3, 0.7
    q, k, v = r.standard_normal((T, dk)), r.standard_normal((T, dk)), r.standard_normal((T, dv))
    o_ref, S_ref = ridge.ridge_atq(q, k, v, lam)
    wk = ridge.atk_write_keys(k, lam)
    S = np.zeros((dk, dv))
    o = np.zeros((T, dv))
    for t in range(T):
        S, o[t], _ = oracle.recurrence_step(S, q[t], k[t], v[t], np.array(1.0), wk[t])
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(S, S_ref, rtol=1e-10, atol=1e-11)


def test_diagonal_counterexample():
    g = golden("ridge_diagonal_counterexample.json")
    k = np.array([g["k1"]])
    v = np.array([g["v1"]])
    S_atq = ridge.diagonal_atq_state(k, v, g["lambda"])
    np.testing.assert_allclose(S_atq, g["diagonal_atq_S1_entry"] * np.ones((2, 2)), atol=1e-15)
    wk = ridge.diagonal_atk_write_keys(k, g["lambda"])
    S_atk, _, _ = oracle.recurrence_step(np.zeros((2, 2)), k[0], k[0], v[0], np.array(1.0), wk[0])
    np.testing.assert_allclose(S_atk, g["diagonal_atk_S1_entry"] * np.ones((2, 2)), atol=1e-15)
    _, S_exact = ridge.ridge_atq(k, k, v, g["lambda"])
    np.testing.assert_allclose(S_exact, S_atk, atol=1e-15)


# ------------------------------------------------------------------ P5: Kalman scalar example

def test_kalman_scalar_gain_example():
    g = golden("kalman_scalar_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"]
    for p_hat, expect in g["gain_at_predicted_variance"].items():
        kap = oracle.kdn_gain(np.array([float(p_hat)]), np.array([g["k"]]), np.array(g["r"]))
        assert kap[0] == pytest.approx(expect, abs=tol)


def test_kalman_repeated_observation_variance():
    """D = 1, Omega = 0, p_0 = 1, k = r = 1: p_n = 1/(n+1) (KDN notes section 2.2)."""
    n = 50
    ones = np.ones((1, n, 1, 1))
    o, S, p = oracle.tokenwise(ones, ones, ones, np.zeros((1, n, 1, 1)), "kdn",
                               omega=np.zeros((1, n, 1, 1)), r=np.ones((1, n, 1)), info_scale=1.0)
    assert p[0, 0, 0] == pytest.approx(1.0 / (n + 1), rel=1e-13)
    for m in (1, 2, 7):
        _, _, pm = oracle.tokenwise(ones[:, :m], ones[:, :m], ones[:, :m], np.zeros((1, m, 1, 1)),
                                    "kdn", omega=np.zeros((1, m, 1, 1)), r=np.ones((1, m, 1)))
        assert pm[0, 0, 0] == pytest.approx(1.0 / (m + 1), rel=1e-14)


def test_diagonal_kdn_equals_exact_kalman_for_axis_keys():
    """With one-hot keys, diagonal decay and diagonal process noise the exact
    posterior covariance stays diagonal, so Diagonal KDN with mu = 1 equals the
    dense Kalman filter (KDN notes Eqs. (12)-(17) vs Eqs. (23)-(30))."""
    r = rng(6)
    T, dk, dv = 30, 5, 3
    k = np.zeros((T, dk))
    k[np.arange(T), r.integers(0, dk, T)] = r.uniform(0.5, 2.0, T)
    q, v = r.standard_normal((T, dk)), r.standard_normal((T, dv))
    alpha = np.exp(-r.uniform(0.0, 0.5, (T, dk)))
    omega = r.uniform(0.0, 0.2, (T, dk))
    rr = r.uniform(0.2, 2.0, T)
    p0 = r.uniform(0.5, 1.5, dk)
    o_ref, S_ref, P_ref, kap_ref = ridge.dense_kalman(q, k, v, alpha, omega, rr, np.diag(p0))
    o, S, p, tr = oracle.tokenwise(q[None, :, None], k[None, :, None], v[None, :, None],
                                   np.log(alpha)[None, :, None], "kdn", omega=omega[None, :, None],
                                   r=rr[None, :, None], info_scale=1.0, aux0=p0[None, None],
                                   return_trace=True)
    np.testing.assert_allclose(tr["w"][0, :, 0], kap_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o[0, :, 0], o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(p[0, 0], np.diag(P_ref), rtol=1e-12)


# ------------------------------------------------------------------ P6: information scaling

def test_information_scaling_example():
    g = golden("information_scaling_example.json")
    m = g["m"]
    k = np.full(m, 1.0 / math.sqrt(m))
    p_hat = np.full(m, g["p"])
    tol = 0.5 * 10 ** -g["printed_decimals"]
    v1 = np.sum(k * k * oracle.kdn_variance_update(p_hat, k, np.array(g["r"]), 1.0))
    vm = np.sum(k * k * oracle.kdn_variance_update(p_hat, k, np.array(g["r"]), float(m)))
    assert v1 == pytest.approx(g["V_proj_mu_1_printed"], abs=tol)
    assert v1 == pytest.approx(m / (m + 1.0), rel=1e-14)
    assert vm == pytest.approx(g["V_proj_mu_m"], abs=1e-15)
    # exact directional variance r p/(r + p) of the dense posterior along k
    P_star = np.linalg.inv(np.diag(1.0 / p_hat) + np.outer(k, k) / g["r"])
    assert k @ P_star @ k == pytest.approx(g["V_exact"], rel=1e-12)


# ------------------------------------------------------------------ P7: reductions

def test_kdn_with_constant_variance_is_kla():
    """p^ = b on every channel and r = eps b turns the Kalman gain into the
    Kaczmarz step with eta = 1 (KDN notes section 3, Eqs. (18)-(20)).  p^ is held
    at b by mu = 0, channel-uniform decay and omega = b (1 - alpha^2)."""
    d = random_inputs("kla", seed=7, B=1, T=25, H=2, dk=6, dv=4)
    b, eps = 0.8, 1e-3
    B_, T, H, dk = d["k"].shape
    la = d["log_alpha"]
    la_c = np.repeat(la[..., None], dk, axis=-1)
    omega = b * (1 - np.exp(2 * la_c))
    o_kdn, S_kdn, p = oracle.tokenwise(d["q"], d["k"], d["v"], la_c, "kdn", omega=omega,
                                       r=np.full((B_, T, H), eps * b), info_scale=0.0,
                                       aux0=np.full((B_, H, dk), b), q_l2norm=True)
    o_kla, S_kla, _ = oracle.tokenwise(d["q"], d["k"], d["v"], la, "kla", eta=np.ones((B_, T, H)),
                                       eps=eps, q_l2norm=True)
    np.testing.assert_allclose(o_kdn, o_kla, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S_kdn, S_kla, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(p, b, rtol=1e-12)


def test_kaczmarz_projection_is_minimum_change():
    """eta = 1, eps = 0, no decay: each write makes S^T k = v hold and is the
    minimum-Frobenius change doing so (KLA notes section 2.2, Eqs. (1)-(2)),
    checked against numpy's least-squares minimum-norm solution."""
    r = rng(8)
    T, dk, dv = 12, 7, 3
    k, v, q = r.standard_normal((T, dk)), r.standard_normal((T, dv)), r.standard_normal((T, dk))
    S = r.standard_normal((dk, dv))
    for t in range(T):
        w = oracle.kla_write(k[t], np.array(1.0), 0.0)
        S_new, _, e = oracle.recurrence_step(S, q[t], k[t], v[t], np.array(1.0), w)
        np.testing.assert_allclose(S_new.T @ k[t], v[t], atol=1e-12)
        delta, *_ = np.linalg.lstsq(k[t][None, :], e[None, :], rcond=None)
        np.testing.assert_allclose(S_new - S, delta, atol=1e-12)
        S = S_new


def test_orthonormal_keys_read_back_exactly():
    """Writes along orthogonal keys do not interfere (KLA notes section 2.4, last
    paragraph): with eta = 1, eps = 0, alpha = 1 every stored pair reads back."""
    r = rng(9)
    dk, dv = 8, 5
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = (Qm.T * r.uniform(0.5, 3.0, dk)[:, None])       # orthogonal, unequal norms
    v = r.standard_normal((dk, dv))
    S = np.zeros((dk, dv))
    for t in range(dk):
        w = oracle.kla_write(k[t], np.array(1.0), 0.0)
        S, _, _ = oracle.recurrence_step(S, k[t], k[t], v[t], np.array(1.0), w)
    np.testing.assert_allclose(k @ S, v, atol=1e-12)


def test_gdn_without_decay_is_deltanet_contraction():
    """log alpha = 0 gives DeltaNet; re-reading gives (1 - beta ||k||^2) e (KLA notes Eq. (5) line 1)."""
    d = random_inputs("gdn", seed=10, B=1, T=9, H=1, dk=5, dv=3)
    d["log_alpha"] = np.zeros_like(d["log_alpha"])
    _, S, _, tr = call(oracle.tokenwise, "gdn", d, return_trace=True)
    k = d["k"][0, :, 0]
    S_t = np.zeros((5, 3))
    for t in range(9):
        S_t, _, e = oracle.recurrence_step(S_t, k[t], k[t], d["v"][0, t, 0], np.array(1.0), tr["w"][0, t, 0])
        beta = d["eta"][0, t, 0]
        np.testing.assert_allclose(d["v"][0, t, 0] - S_t.T @ k[t], (1 - beta * k[t] @ k[t]) * e, atol=1e-11)


# ------------------------------------------------------------------ KDA / PKDA reductions

@pytest.mark.parametrize("pair", [("kda", "gdn"), ("pkda", "pgdn")])
def test_per_channel_decay_uniform_across_channels_reduces(pair):
    """KDA with alpha_t the same on every channel is Gated DeltaNet (KDN notes
    section 1, table: D_t = diag(alpha_t) vs alpha_t I, same write beta k), and
    PKDA so reduces to PGDN (PDN notes section 2.5, the unified form)."""
    vec, sca = pair
    d = random_inputs(vec, B=2, T=29, H=2, dk=5, dv=3, seed=21)
    la = d["log_alpha"][..., 0]
    d["log_alpha"] = np.repeat(la[..., None], 5, axis=-1)
    s = dict(d, log_alpha=la)
    r = rng(22)
    S0 = r.standard_normal((2, 2, 5, 3))
    aux0 = r.uniform(0, 2, (2, 2, 5)) if vec == "pkda" else None
    for fn in (oracle.tokenwise, lambda *a, **k: oracle.chunkwise(*a, chunk=8, **k)):
        o1, S1, a1 = call(fn, vec, d, S0=S0, aux0=aux0, q_l2norm=True)
        o2, S2, a2 = call(fn, sca, s, S0=S0, aux0=aux0, q_l2norm=True)
        np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S1, S2, rtol=1e-12, atol=1e-13)
        if a1 is not None:
            np.testing.assert_allclose(a1, a2, rtol=1e-13)


@pytest.mark.parametrize("variant", ["kda", "pkda"])
def test_per_channel_decay_scales_key_rows(variant):
    """With nothing written (eta = 0) the memory only decays: S_t = D_t ... D_1 S_0
    with D = diag(alpha) acting on the key index (KDN notes section 1), so the
    read is o_t[v] = sum_i q_t[i] prod_{s <= t} alpha_s[i] S_0[i, v].  dk != dv,
    so decaying the value index instead fails."""
    d = random_inputs(variant, B=1, T=11, H=1, dk=4, dv=6, seed=23)
    d["eta"] = np.zeros_like(d["eta"])
    S0 = rng(24).standard_normal((1, 1, 4, 6))
    cum = np.exp(np.cumsum(d["log_alpha"][0, :, 0], axis=0))          # [T, dk]
    expect = np.einsum("ti,ti,iv->tv", d["q"][0, :, 0], cum, S0[0, 0])
    for fn in (oracle.tokenwise, lambda *a, **k: oracle.chunkwise(*a, chunk=4, **k)):
        o, S, _ = call(fn, variant, d, S0=S0)
        np.testing.assert_allclose(o[0, :, 0], expect, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(S[0, 0], cum[-1][:, None] * S0[0, 0], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ isotropic KDN

@pytest.mark.parametrize("mu", [1.0, 3.0])
def test_isotropic_kdn_with_one_channel_is_diagonal_kdn(mu):
    """With dk = 1 the isotropic and diagonal filters are the same scalar Kalman
    filter (KDN notes section 7 vs Eqs. (23)-(30), (60)-(65)): a = alpha^2,
    beta k = p^ k/(r + p^ k^2), u = mu k^2 / r."""
    d = random_inputs("kdn", B=2, T=23, H=2, dk=1, dv=3, seed=31)
    S0 = rng(32).standard_normal((2, 2, 1, 3))
    p0 = rng(33).uniform(0.5, 1.5, (2, 2, 1))
    o1, S1, p1 = call(oracle.tokenwise, "kdn", d, S0=S0, aux0=p0, info_scale=mu)
    di = dict(d, omega=d["omega"][..., 0])
    o2, S2, b2 = call(oracle.tokenwise, "ikdn", di, S0=S0, aux0=p0[..., 0], info_scale=mu)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S2, S1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(b2, p1[..., 0], rtol=1e-13)


def test_isotropic_kdn_scalar_gain_example():
    """The pages' scalar Kalman gains (k = r = 1: p^ = 9 -> 0.9, p^ = 0.1 -> 0.0909)
    hold for the isotropic gain beta = b^/(r + b^ ||k||^2) (KDN notes section 7)."""
    g = golden("kalman_scalar_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"]
    for b_hat, expect in g["gain_at_predicted_variance"].items():
        w = oracle.ikdn_gain(np.array(float(b_hat)), np.array([g["k"]]), np.array(g["r"]))
        assert w[0] == pytest.approx(expect, abs=tol)


def test_isotropic_kdn_unit_keys_at_mu_dk():
    """With unit keys and mu = dk the update weight is u = 1/r, so every step
    gives b = b^/(1 + b^/r) (KDN notes section 7, the remark after Eq. (40))."""
    d = random_inputs("ikdn", B=1, T=15, H=2, dk=6, dv=3, seed=34)
    d["k"] = oracle.l2normalize(d["k"])
    B, T, H, dk = d["k"].shape
    b = np.ones((B, H))
    for t in range(T):
        one = {key: (val[:, t:t + 1] if val.ndim >= 3 else val) for key, val in d.items()}
        _, _, b_next = call(oracle.tokenwise, "ikdn", one, aux0=b, info_scale=float(dk))
        b_hat = np.mean(np.exp(2 * d["log_alpha"][:, t]), axis=-1) * b + d["omega"][:, t]
        np.testing.assert_allclose(b_next, b_hat / (1 + b_hat / d["r"][:, t]), rtol=1e-14)
        b = b_next


def test_isotropic_kdn_predicts_with_the_mean_squared_decay():
    """The trace projection: with no process noise and no information (r large)
    the variance only decays, b_t = b_0 prod_s mean_i alpha_{s,i}^2 -- neither the
    squared mean decay nor the mean decay (KDN notes section 7, Eq. (40) first line)."""
    d = random_inputs("ikdn", B=1, T=5, H=1, dk=5, dv=2, seed=35)
    d["omega"] = np.zeros_like(d["omega"])
    d["r"] = np.full_like(d["r"], 1e300)
    _, _, b = call(oracle.tokenwise, "ikdn", d, aux0=np.full((1, 1), 2.0))
    alpha = np.exp(d["log_alpha"][0, :, 0])                       # [T, dk]
    expect = 2.0 * np.prod(np.mean(alpha * alpha, axis=1))
    assert b[0, 0] == pytest.approx(expect, rel=1e-12)
    other = 2.0 * np.prod(np.mean(alpha, axis=1) ** 2)
    assert abs(other - expect) > 1e-3 * expect


# ------------------------------------------------------------------ exact Kalman memory

def test_exact_kalman_tokenwise_matches_dense_side_oracle():
    """The batched tokenwise exact Kalman variant equals the independently written
    single-head dense filter (KDN notes section 2.2, Eqs. (12)-(17)) on random
    data, head by head, from a random SPD P_0."""
    r_ = rng(41)
    B, T, H, dk, dv = 2, 13, 2, 5, 3
    d = random_inputs("kdn", B=B, T=T, H=H, dk=dk, dv=dv, seed=42)
    A = r_.standard_normal((B, H, dk, dk))
    P0 = A @ np.swapaxes(A, -1, -2) / dk + 0.5 * np.eye(dk)
    o, S, P = call(oracle.tokenwise, "ekdn", d, aux0=P0)
    for b in range(B):
        for h in range(H):
            o_r, S_r, P_r, _ = ridge.dense_kalman(d["q"][b, :, h], d["k"][b, :, h], d["v"][b, :, h],
                                                  np.exp(d["log_alpha"][b, :, h]),
                                                  d["omega"][b, :, h], d["r"][b, :, h], P0[b, h])
            np.testing.assert_allclose(o[b, :, h], o_r, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(S[b, h], S_r, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(P[b, h], P_r, rtol=1e-11, atol=1e-12)


def test_exact_kalman_with_axis_keys_is_diagonal_kdn():
    """Keys along coordinate axes keep a diagonal covariance diagonal, so the exact
    filter and Diagonal KDN (mu = 1) agree (KDN notes Eqs. (12)-(17) vs (23)-(30))."""
    r_ = rng(43)
    B, T, H, dk, dv = 1, 17, 2, 4, 3
    d = random_inputs("kdn", B=B, T=T, H=H, dk=dk, dv=dv, seed=44)
    axes = r_.integers(0, dk, (B, T, H))
    d["k"] = np.eye(dk)[axes] * r_.uniform(0.5, 2.0, (B, T, H, 1))
    p0 = r_.uniform(0.5, 1.5, (B, H, dk))
    o1, S1, p1 = call(oracle.tokenwise, "kdn", d, aux0=p0, info_scale=1.0)
    o2, S2, P2 = call(oracle.tokenwise, "ekdn", d, aux0=p0[..., :, None] * np.eye(dk))
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(np.diagonal(P2, axis1=-2, axis2=-1), p1, rtol=1e-12)
    np.testing.assert_allclose(P2 - np.diagonal(P2, axis1=-2, axis2=-1)[..., None] * np.eye(dk), 0,
                               atol=1e-15)


def test_exact_kalman_scalar_gain_example():
    """dk = 1: the pages' scalar gains (k = r = 1: P^ = 9 -> 0.9, 0.1 -> 0.0909)."""
    g = golden("kalman_scalar_example.json")
    tol = 0.5 * 10 ** -g["printed_decimals"]
    for p_hat, expect in g["gain_at_predicted_variance"].items():
        kap = oracle.ekdn_gain(np.array([[float(p_hat)]]), np.array([g["k"]]), np.array(g["r"]))
        assert kap[0] == pytest.approx(expect, abs=tol)


def test_exact_kalman_resume_split_equals_whole():
    """The state (S, P) is the whole checkpoint: fwd(T) = fwd(T1) then fwd(T2)."""
    d = random_inputs("kdn", B=1, T=20, H=2, dk=4, dv=3, seed=45)
    o, S, P = call(oracle.tokenwise, "ekdn", d, q_l2norm=True)
    head = {k: (v[:, :9] if v.ndim >= 3 else v) for k, v in d.items()}
    tail = {k: (v[:, 9:] if v.ndim >= 3 else v) for k, v in d.items()}
    o1, S1, P1 = call(oracle.tokenwise, "ekdn", head, q_l2norm=True)
    o2, S2, P2 = call(oracle.tokenwise, "ekdn", tail, S0=S1, aux0=P1, q_l2norm=True)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(P2, P, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ P8: tokenwise == chunkwise

CASES = [  # (T, dk, dv, chunk)
    (1, 4, 3, 4), (2, 2, 2, 1), (3, 4, 3, 2), (17, 4, 5, 4), (63, 8, 4, 16), (64, 8, 4, 16),
    (65, 8, 4, 16), (130, 4, 3, 64), (40, 2, 2, 64), (33, 8, 8, 32),
]


@pytest.mark.parametrize("variant", oracle.VARIANTS)
@pytest.mark.parametrize("T,dk,dv,chunk", CASES)
def test_tokenwise_equals_chunkwise(variant, T, dk, dv, chunk):
    d = random_inputs(variant, B=1, T=T, H=2, dk=dk, dv=dv, seed=T * 31 + dk)
    r = rng(T)
    S0 = r.standard_normal((1, 2, dk, dv))
    aux0 = {"pgdn": r.uniform(0, 2, (1, 2, dk)), "pkda": r.uniform(0, 2, (1, 2, dk)),
            "kdn": r.uniform(0.5, 1.5, (1, 2, dk)), "ikdn": r.uniform(0.5, 1.5, (1, 2))}.get(variant)
    kw = dict(S0=S0, aux0=aux0, q_l2norm=True,
              k_l2norm=(variant in ("pgdn", "pkda", "kdn", "ikdn")), eps=1e-6)
    o1, S1, a1 = call(oracle.tokenwise, variant, d, **kw)
    o2, S2, a2 = call(oracle.chunkwise, variant, d, chunk=chunk, **kw)
    scale = max(1.0, np.abs(o1).max())
    np.testing.assert_allclose(o2, o1, atol=1e-10 * scale, rtol=1e-9)
    np.testing.assert_allclose(S2, S1, atol=1e-10 * max(1.0, np.abs(S1).max()), rtol=1e-9)
    if a1 is not None:
        np.testing.assert_allclose(a2, a1, rtol=1e-11)


def test_chunkwise_strong_decay_matches_tokenwise():
    """The workloads' decay (mean log alpha ~ -2.2 per token) underflows gamma over
    a 64-token chunk; ratios from log differences keep the chunk form exact."""
    for variant in ("kla", "kdn"):
        d = random_inputs(variant, B=1, T=150, H=1, dk=8, dv=4, seed=11, decay_shift=2.0)
        o1, S1, _ = call(oracle.tokenwise, variant, d, q_l2norm=True, eps=1e-6)
        o2, S2, _ = call(oracle.chunkwise, variant, d, chunk=64, q_l2norm=True, eps=1e-6)
        np.testing.assert_allclose(o2, o1, atol=1e-10 * np.abs(o1).max(), rtol=1e-8)


def test_chunked_gain_scans_match_sequential():
    """PGDN's chunked statistic (PDN notes section 2.6) and the Moebius prefix
    products (KDN notes Eqs. (32)-(39)) equal the token-by-token recursions."""
    r = rng(12)
    C, dk = 40, 6
    k = r.standard_normal((C, dk))
    aP, bP = 1 / (1 + np.exp(-(r.standard_normal(C) + 3))), r.uniform(0, 1, C)
    A_in = r.uniform(0, 2, dk)
    A_seq, A = [], A_in
    for t in range(C):
        A = oracle.pgdn_stat_update(A, k[t], np.array(aP[t]), np.array(bP[t]))
        A_seq.append(A)
    np.testing.assert_allclose(oracle.pgdn_stat_chunk(A_in, k * k, np.log(aP), bP), A_seq, rtol=1e-12)

    alpha, omega = np.exp(-r.uniform(0, 3, (C, dk))), r.uniform(0, 0.3, (C, dk))
    rr = r.uniform(0.2, 2, C)
    mu = 3.0
    u = (mu / rr)[:, None] * k * k
    p_in = r.uniform(0.5, 2, dk)
    p_prev, p_post = oracle.kdn_mobius_chunk(p_in, alpha, omega, u)
    p = p_in
    for t in range(C):
        np.testing.assert_allclose(p_prev[t], p, rtol=1e-12)
        p = oracle.kdn_variance_update(oracle.kdn_predict(p, alpha[t], omega[t]), k[t], np.array(rr[t]), mu)
        np.testing.assert_allclose(p_post[t], p, rtol=1e-12)


def test_mobius_product_is_ordered():
    """Associative but not commutative (KDN notes section 6): reversing the token
    order changes p."""
    r = rng(13)
    C, dk = 6, 3
    alpha, omega = np.exp(-r.uniform(0, 2, (C, dk))), r.uniform(0.1, 0.5, (C, dk))
    u = r.uniform(0.5, 2, (C, dk))
    _, fwd = oracle.kdn_mobius_chunk(np.ones(dk), alpha, omega, u)
    _, rev = oracle.kdn_mobius_chunk(np.ones(dk), alpha[::-1], omega[::-1], u[::-1])
    assert np.abs(fwd[-1] - rev[-1]).max() > 1e-3


# ------------------------------------------------------------------ P9: resume

@pytest.mark.parametrize("variant", oracle.VARIANTS)
def test_resume_split_equals_whole(variant):
    """fwd(T) = fwd(T1) then fwd(T2, init = final state): the recurrent state is
    the whole checkpoint (KDN notes section 8: training scan and token-by-token
    inference are one recurrence)."""
    d = random_inputs(variant, B=1, T=50, H=2, dk=4, dv=3, seed=14)
    kw = dict(q_l2norm=True, eps=1e-6)
    o, S, a = call(oracle.chunkwise, variant, d, chunk=16, **kw)
    cut = 21
    head = {k: (v[:, :cut] if v.ndim >= 3 else v) for k, v in d.items()}
    tail = {k: (v[:, cut:] if v.ndim >= 3 else v) for k, v in d.items()}
    o1, S1, a1 = call(oracle.chunkwise, variant, head, chunk=16, **kw)
    # continue with the tokenwise form (the decode path) from the chunkwise state
    o2, S2, a2 = call(oracle.tokenwise, variant, tail, S0=S1, aux0=a1, **kw)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S2, S, rtol=1e-9, atol=1e-11)


# ------------------------------------------------------------------ backward (reverse mode)

from oracle import backward as obw  # noqa: E402


@pytest.mark.parametrize("variant", obw.GRAD_VARIANTS)
@pytest.mark.parametrize("norm", [False, True])
def test_backward_matches_central_differences(variant, norm):
    """Every gradient of L = <dO, O> + <dS_T, S_T> + <daux_T, aux_T> (q, k, v,
    log alpha, the variant's gates, S_0 and the gain state's initial value)
    equals the central difference of the forward oracle, element by element:
    the reverse sweep is pinned to the independently written forward."""
    r = rng(60)
    B, T, H, dk, dv = 1, 6, 2, 3, 2
    d = random_inputs("kdn" if variant == "ekdn" else variant, B=B, T=T, H=H, dk=dk, dv=dv, seed=61)
    d["S0"] = r.standard_normal((B, H, dk, dv))
    if variant in ("pgdn", "pkda"):
        d["aux0"] = r.uniform(0.5, 2.0, (B, H, dk))
    elif variant == "kdn":
        d["aux0"] = r.uniform(0.5, 1.5, (B, H, dk))
    elif variant == "ikdn":
        d["aux0"] = r.uniform(0.5, 1.5, (B, H))
    elif variant == "ekdn":   # an SPD covariance
        A = r.standard_normal((B, H, dk, dk))
        d["aux0"] = A @ np.swapaxes(A, -1, -2) / dk + 0.5 * np.eye(dk)
    dO = r.standard_normal((B, T, H, dv))
    dS = r.standard_normal((B, H, dk, dv))
    daux = r.standard_normal(d["aux0"].shape) if "aux0" in d else None
    flags = dict(q_l2norm=norm, k_l2norm=norm, eps=1e-6)
    gate_keys = [kk for kk in ("eta", "alphaP", "betaP", "mu", "omega", "r") if kk in d]

    def loss(dd):
        o, S, aux = oracle.tokenwise(dd["q"], dd["k"], dd["v"], dd["log_alpha"], variant,
                                     S0=dd["S0"], aux0=dd.get("aux0"),
                                     **{kk: dd[kk] for kk in gate_keys}, **flags)
        out = float(np.sum(dO * o) + np.sum(dS * S))
        return out + (float(np.sum(daux * aux)) if daux is not None else 0.0)

    g = obw.tokenwise_backward(d["q"], d["k"], d["v"], d["log_alpha"], variant, dO, dS,
                               S0=d["S0"], aux0=d.get("aux0"), daux_T=daux,
                               **{kk: d[kk] for kk in gate_keys}, **flags)
    names = {"q": "dq", "k": "dk", "v": "dv", "log_alpha": "dlog_alpha", "eta": "deta",
             "alphaP": "dalphaP", "betaP": "dbetaP", "mu": "dmu", "omega": "domega", "r": "dr",
             "S0": "dS0", "aux0": "daux0"}
    h = 1e-6
    for name, key in names.items():
        if name not in d:
            continue
        num = np.zeros_like(d[name])
        for idx in np.ndindex(d[name].shape):
            dp = {kk: vv.copy() for kk, vv in d.items()}
            dm = {kk: vv.copy() for kk, vv in d.items()}
            dp[name][idx] += h
            dm[name][idx] -= h
            num[idx] = (loss(dp) - loss(dm)) / (2 * h)
        np.testing.assert_allclose(g[key], num, rtol=1e-5, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("variant", ["gdn", "kla", "kda", "pgdn", "pkda", "kdn", "ikdn"])
@pytest.mark.parametrize("T,chunk", [(1, 4), (7, 4), (16, 8), (13, 64), (21, 2)])
def test_chunkwise_backward_equals_tokenwise_backward(variant, T, chunk):
    """The chunk-by-chunk reverse sweep through Eqs. (7)-(9) (the form a kernel
    follows), with the gain recursion's reverse sweep from dL/dw, gives the
    tokenwise reverse sweep's gradients to rounding."""
    r = rng(70 + T)
    B, H, dk, dv = 2, 2, 4, 3
    d = random_inputs(variant, B=B, T=T, H=H, dk=dk, dv=dv, seed=71 + T)
    S0 = r.standard_normal((B, H, dk, dv))
    dO = r.standard_normal((B, T, H, dv))
    dS = r.standard_normal((B, H, dk, dv))
    aux_shape = {"pgdn": (B, H, dk), "pkda": (B, H, dk), "kdn": (B, H, dk), "ikdn": (B, H)}.get(variant)
    aux0 = r.uniform(0.5, 1.5, aux_shape) if aux_shape else None
    daux = r.standard_normal(aux_shape) if aux_shape else None
    gates = {kk: d[kk] for kk in ("eta", "alphaP", "betaP", "mu", "omega", "r") if kk in d}
    kw = dict(S0=S0, aux0=aux0, daux_T=daux, q_l2norm=True,
              k_l2norm=(variant not in ("gdn", "kla")), eps=1e-6, **gates)
    g1 = obw.tokenwise_backward(d["q"], d["k"], d["v"], d["log_alpha"], variant, dO, dS, **kw)
    g2 = obw.chunkwise_backward(d["q"], d["k"], d["v"], d["log_alpha"], variant, chunk, dO, dS, **kw)
    assert set(g1) == set(g2), (sorted(g1), sorted(g2))
    for key in g1:
        np.testing.assert_allclose(g2[key], g1[key], rtol=1e-9, atol=1e-11, err_msg=key)
