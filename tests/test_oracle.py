"""Pins of the fp64 oracle against what the paper and the mathematics fix.

Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
Probabilistic Latent Routing" (Huang & Raza, 2026).  The paper prints no
worked numerical example of Gamma or O, so the oracle is pinned by:

* a textbook routine: scipy's multivariate normal log-density with a diagonal
  covariance, plus log-priors, softmaxed (Eq. 2, 3, 14, 15, 16);
* the explicit N x N affinity of Eq. (9)-(10) (bidirectional) and Eq. (9b)-(10b)
  (causal), built by brute force and applied to V;
* closed forms: K = 1 (prefix) mean, identical components, one-hot limit;
* invariants: rows of Gamma on the simplex (section 3.2), non-negative
  affinity of rank <= K (Eq. 23), sum_k Z_k = N (Eq. 6), convex combinations
  at eps = 0, permutation equivariance, exact prefix causality (section 3.5),
  Theorem 1's Jacobian bound (section 4.3).

A non-negligible eps is used where the test must pin where eps enters.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle

RNG = np.random.default_rng(1234)


def make(N=40, d=5, K=7, dv=6, mu_std=1.0, rho_std=0.5, seed=0):
    r = np.random.default_rng(seed)
    return dict(
        Qx=r.normal(size=(N, d)), Kx=r.normal(size=(N, d)), V=r.normal(size=(N, dv)),
        mu=mu_std * r.normal(size=(K, d)), omega=rho_std * r.normal(size=(K, d)),
        alpha=r.normal(size=(K,)),
    )


def textbook_scores(X, mu, omega, alpha, var_floor):
    """log pi_k + log N(x | mu_k, diag(var_k)) with scipy's density routine."""
    var = np.logaddexp(0.0, omega) + var_floor          # softplus by a different formula
    logpi = special.log_softmax(alpha)
    cols = [stats.multivariate_normal(mean=mu[k], cov=np.diag(var[k])).logpdf(X)
            for k in range(mu.shape[0])]
    return np.stack([np.atleast_1d(c) for c in cols], axis=1) + logpi[None, :]


def textbook_gamma(X, mu, omega, alpha, var_floor):
    return special.softmax(textbook_scores(X, mu, omega, alpha, var_floor), axis=1)


def brute_force(Qx, Kx, V, mu, omega, alpha, var_floor, eps, causal):
    """Eq. (9)-(10) / (9b)-(10b): explicit affinity, row-normalised, applied to V."""
    gq = textbook_gamma(Qx, mu, omega, alpha, var_floor)
    gk = textbook_gamma(Kx, mu, omega, alpha, var_floor)
    At = gq @ gk.T
    if causal:
        At = np.tril(At)
    A = At / (At.sum(axis=1, keepdims=True) + eps)
    return A @ V, A, At


# ---------------------------------------------------------------- responsibilities

@pytest.mark.parametrize("d,K,floor", [(5, 7, 1e-4), (1, 3, 1e-2), (16, 8, 1e-4), (3, 1, 1e-4)])
def test_scores_match_textbook_density(d, K, floor):
    p = make(N=33, d=d, K=K, rho_std=1.5, seed=d * 10 + K)
    s = oracle.scores(p["Qx"], p["mu"], p["omega"], p["alpha"], floor)
    ref = textbook_scores(p["Qx"], p["mu"], p["omega"], p["alpha"], floor)
    np.testing.assert_allclose(s, ref, rtol=0, atol=1e-10 * max(1.0, np.abs(ref).max()))


def test_responsibilities_match_textbook_posterior():
    p = make(N=64, d=6, K=9, mu_std=2.0, rho_std=1.0, seed=7)
    g = oracle.responsibilities(p["Kx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    ref = textbook_gamma(p["Kx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    np.testing.assert_allclose(g, ref, rtol=0, atol=1e-13)


def test_responsibilities_are_on_the_simplex():
    p = make(N=200, d=8, K=16, mu_std=3.0, seed=3)
    g = oracle.responsibilities(p["Qx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    assert (g >= 0).all()
    np.testing.assert_allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_responsibilities_component_permutation_and_prior_shift():
    p = make(N=50, d=4, K=6, seed=11)
    g = oracle.responsibilities(p["Qx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    perm = RNG.permutation(6)
    gp = oracle.responsibilities(p["Qx"], p["mu"][perm], p["omega"][perm], p["alpha"][perm], 1e-4)
    np.testing.assert_allclose(gp, g[:, perm], rtol=0, atol=1e-14)
    gs = oracle.responsibilities(p["Qx"], p["mu"], p["omega"], p["alpha"] + 3.7, 1e-4)
    np.testing.assert_allclose(gs, g, rtol=0, atol=1e-14)


def test_variance_floor_enters_the_density():
    # omega -> -inf makes softplus -> 0, so the variance is the floor alone.
    p = make(N=10, d=3, K=2, seed=5)
    om = np.full_like(p["omega"], -60.0)
    s = oracle.scores(p["Qx"], p["mu"], om, p["alpha"], 0.25)
    x, mu = p["Qx"], p["mu"]
    ref = (special.log_softmax(p["alpha"])[None, :] - 0.5 * 3 * np.log(2 * np.pi)
           - 0.5 * 3 * np.log(0.25)
           - 0.5 * ((x[:, None, :] - mu[None, :, :]) ** 2).sum(-1) / 0.25)
    np.testing.assert_allclose(s, ref, rtol=1e-13, atol=1e-12)


# ---------------------------------------------------------------- forward vs brute force

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,K,dv,eps", [(1, 3, 4, 2, 1e-6), (17, 5, 7, 6, 1e-6),
                                          (128, 16, 8, 32, 1e-6), (300, 4, 12, 5, 0.3),
                                          (512, 8, 3, 4, 1e-3)])
def test_forward_matches_explicit_affinity(causal, N, d, K, dv, eps):
    p = make(N=N, d=d, K=K, dv=dv, seed=N + K)
    out = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                              1e-4, eps, causal)
    ref, _, _ = brute_force(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                            1e-4, eps, causal)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_affinity_is_nonnegative_and_rank_at_most_K():
    p = make(N=64, d=6, K=8, seed=21)
    gq = oracle.responsibilities(p["Qx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    gk = oracle.responsibilities(p["Kx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    At = gq @ gk.T
    assert (At >= 0).all()
    sv = np.linalg.svd(At, compute_uv=False)
    assert sv[8] / sv[0] < 1e-12
    A = At / (At.sum(1, keepdims=True) + 1e-6)
    sv = np.linalg.svd(A, compute_uv=False)
    assert sv[8] / sv[0] < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_memory_mass_sums_to_sequence_length(causal):
    p = make(N=97, d=5, K=11, seed=2)
    _, Vt, Z = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                                   1e-4, 1e-6, causal, return_memory=True)
    assert abs(Z.sum() - 97) < 1e-11
    gk = textbook_gamma(p["Kx"], p["mu"], p["omega"], p["alpha"], 1e-4)
    np.testing.assert_allclose(Vt, gk.T @ p["V"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Z, gk.sum(0), rtol=1e-12, atol=1e-12)


def test_causal_row_equals_bidirectional_on_the_prefix():
    # Eq. (8b) for row i is Eq. (8) on the sequence truncated after i.
    p = make(N=40, d=4, K=5, dv=3, seed=9)
    oc = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                             1e-4, 0.05, True)
    for i in (0, 1, 7, 39):
        ob = oracle.forward_head(p["Qx"][:i + 1], p["Kx"][:i + 1], p["V"][:i + 1], p["mu"],
                                 p["omega"], p["alpha"], 1e-4, 0.05, False)
        np.testing.assert_allclose(oc[i], ob[i], rtol=1e-12, atol=1e-13)


def test_causal_prefix_error_is_exactly_zero():
    # Section 5.3 reports a maximum prefix error of zero: rows <= i must not see rows > i.
    p = make(N=60, d=4, K=6, dv=5, seed=31)
    o1 = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                             1e-4, 1e-6, True)
    q = {k: v.copy() for k, v in p.items()}
    q["Qx"][30:] = RNG.normal(size=q["Qx"][30:].shape) * 5
    q["Kx"][30:] = RNG.normal(size=q["Kx"][30:].shape) * 5
    q["V"][30:] = RNG.normal(size=q["V"][30:].shape) * 5
    o2 = oracle.forward_head(q["Qx"], q["Kx"], q["V"], q["mu"], q["omega"], q["alpha"],
                             1e-4, 1e-6, True)
    assert np.array_equal(o1[:30], o2[:30])
    assert not np.allclose(o1[30:], o2[30:])


def test_bidirectional_permutation_equivariance():
    p = make(N=50, d=4, K=6, dv=3, seed=17)
    o = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                            1e-4, 1e-6, False)
    pq, pk = RNG.permutation(50), RNG.permutation(50)
    o2 = oracle.forward_head(p["Qx"][pq], p["Kx"][pk], p["V"][pk], p["mu"], p["omega"],
                             p["alpha"], 1e-4, 1e-6, False)
    np.testing.assert_allclose(o2, o[pq], rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_single_component_is_the_prefix_mean(causal):
    p = make(N=37, d=3, K=1, dv=4, seed=4)
    eps = 0.7   # large, so a misplaced eps shows
    o = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                            1e-4, eps, causal)
    if causal:
        cnt = np.arange(1, 38)[:, None]
        ref = np.cumsum(p["V"], axis=0) / (cnt + eps)
    else:
        ref = np.broadcast_to(p["V"].sum(0) / (37 + eps), o.shape)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_components_give_prior_weights(causal):
    p = make(N=25, d=4, K=5, dv=3, seed=8)
    mu = np.tile(p["mu"][:1], (5, 1))
    om = np.tile(p["omega"][:1], (5, 1))
    pi = special.softmax(p["alpha"])
    g = oracle.responsibilities(p["Qx"], mu, om, p["alpha"], 1e-4)
    np.testing.assert_allclose(g, np.broadcast_to(pi, g.shape), rtol=1e-13, atol=1e-15)
    eps = 0.2
    o = oracle.forward_head(p["Qx"], p["Kx"], p["V"], mu, om, p["alpha"], 1e-4, eps, causal)
    s2 = (pi ** 2).sum()
    if causal:
        cnt = np.arange(1, 26)[:, None]
        ref = s2 * np.cumsum(p["V"], 0) / (cnt * s2 + eps)
    else:
        ref = np.broadcast_to(s2 * p["V"].sum(0) / (25 * s2 + eps), o.shape)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_one_hot_limit_is_the_cluster_mean(causal):
    K, d, N, dv = 4, 4, 48, 3
    mu = 20.0 * np.eye(K, d)
    om = np.full((K, d), -40.0)            # variance -> the floor
    alpha = RNG.normal(size=K)
    r = np.random.default_rng(5)
    zq, zk = r.integers(0, K, N), r.integers(0, K, N)
    V = r.normal(size=(N, dv))
    eps = 0.1
    o = oracle.forward_head(mu[zq], mu[zk], V, mu, om, alpha, 1e-4, eps, causal)
    ref = np.zeros((N, dv))
    for i in range(N):
        js = [j for j in range(N) if zk[j] == zq[i] and (j <= i or not causal)]
        ref[i] = V[js].sum(0) / (len(js) + eps) if js else 0.0
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_eps_gives_convex_combinations(causal):
    p = make(N=80, d=5, K=6, dv=4, seed=13)
    o = oracle.forward_head(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                            1e-4, 0.0, causal)
    _, A, _ = brute_force(p["Qx"], p["Kx"], p["V"], p["mu"], p["omega"], p["alpha"],
                          1e-4, 0.0, causal)
    assert (A >= 0).all()
    np.testing.assert_allclose(A.sum(1), 1.0, rtol=0, atol=1e-12)
    for i in range(80):
        lim = slice(0, i + 1) if causal else slice(None)
        lo, hi = p["V"][lim].min(0), p["V"][lim].max(0)
        assert (o[i] >= lo - 1e-12).all() and (o[i] <= hi + 1e-12).all()
    np.testing.assert_allclose(o, A @ p["V"], rtol=1e-11, atol=1e-12)


def test_theorem1_score_jacobian_bound():
    # Section 4.3, Theorem 1: ||J_s(x)||_2 <= sqrt(K) R / eps_sigma with R = max_k ||x - mu_k||.
    p = make(N=1, d=6, K=5, rho_std=2.0, seed=19)
    floor = 1e-2
    x0 = p["Qx"][0]
    h = 1e-6
    J = np.empty((5, 6))
    for m in range(6):
        e = np.zeros(6)
        e[m] = h
        sp = oracle.scores((x0 + e)[None], p["mu"], p["omega"], p["alpha"], floor)[0]
        sm = oracle.scores((x0 - e)[None], p["mu"], p["omega"], p["alpha"], floor)[0]
        J[:, m] = (sp - sm) / (2 * h)
    var = np.logaddexp(0.0, p["omega"]) + floor
    np.testing.assert_allclose(J, -(x0[None] - p["mu"]) / var, rtol=1e-6, atol=1e-6)
    R = np.linalg.norm(x0[None] - p["mu"], axis=1).max()
    assert np.linalg.norm(J, 2) <= np.sqrt(5) * R / floor


def test_multi_head_driver_matches_per_head():
    B, H, N, d, K, dv = 2, 3, 20, 4, 5, 3
    r = np.random.default_rng(3)
    Qx, Kx = r.normal(size=(B, H, N, d)), r.normal(size=(B, H, N, d))
    V = r.normal(size=(B, H, N, dv))
    mu, om, al = r.normal(size=(H, K, d)), r.normal(size=(H, K, d)), r.normal(size=(H, K))
    for causal in (False, True):
        o = oracle.forward(Qx, Kx, V, mu, om, al, 1e-4, 1e-6, causal, threads=4)
        for b in range(B):
            for h in range(H):
                oh = oracle.forward_head(Qx[b, h], Kx[b, h], V[b, h], mu[h], om[h], al[h],
                                         1e-4, 1e-6, causal)
                assert np.array_equal(o[b, h], oh)


# ---------------------------------------------------------------- diagnostics (section 5.4)

def make_heads(B=2, H=3, N=30, d=5, K=6, seed=7, mu_std=1.0):
    r = np.random.default_rng(seed)
    return dict(Qx=r.normal(size=(B, H, N, d)), mu=mu_std * r.normal(size=(H, K, d)),
                omega=0.5 * r.normal(size=(H, K, d)), alpha=r.normal(size=(H, K)))


def test_diagnostics_match_textbook_head_average():
    # Eq. (24)-(29) from scipy's densities and scipy's entropy routine
    x = make_heads()
    B, H, N, _ = x["Qx"].shape
    K = x["mu"].shape[1]
    gbar = np.zeros((B, N, K))
    for b in range(B):
        for h in range(H):
            gbar[b] += textbook_gamma(x["Qx"][b, h], x["mu"][h], x["omega"][h], x["alpha"][h], 1e-4) / H
    flat = gbar.reshape(B * N, K)
    p_ref = flat.mean(axis=0)
    p, husage, htoken, rmax, z = oracle.diagnostics(x["Qx"], x["mu"], x["omega"], x["alpha"], 1e-4)
    np.testing.assert_allclose(p, p_ref, rtol=1e-10, atol=1e-13)
    assert husage == pytest.approx(stats.entropy(p_ref) / np.log(K), rel=1e-10)
    assert htoken == pytest.approx(np.mean([stats.entropy(row) for row in flat]) / np.log(K), rel=1e-10)
    assert rmax == pytest.approx(flat.max(axis=1).mean(), rel=1e-12)
    assert np.array_equal(z.reshape(-1), flat.argmax(axis=1))


def test_diagnostics_identical_components_are_uniform():
    # identical components and priors: gamma = 1/K everywhere -> p = 1/K, both entropies 1,
    # R_max = 1/K, every argmax tie resolved to component 0
    x = make_heads(K=5)
    x["mu"][:] = x["mu"][:, :1]
    x["omega"][:] = x["omega"][:, :1]
    x["alpha"][:] = 0.3
    p, husage, htoken, rmax, z = oracle.diagnostics(x["Qx"], x["mu"], x["omega"], x["alpha"], 1e-4)
    np.testing.assert_allclose(p, 0.2, rtol=1e-12)
    assert husage == pytest.approx(1.0, rel=1e-12)
    assert htoken == pytest.approx(1.0, rel=1e-12)
    assert rmax == pytest.approx(0.2, rel=1e-12)
    assert (z == 0).all()


def test_diagnostics_one_hot_limit():
    # tokens on well-separated component means with tiny variances: gamma is one-hot, so
    # z is the planted component, p its frequency, H_usage that frequency's entropy,
    # H_token = 0 and R_max = 1
    B, H, N, d, K = 1, 2, 24, 3, 4
    r = np.random.default_rng(3)
    mu1 = 10.0 * np.eye(K, d) + np.arange(K)[:, None] * 7.0
    mu = np.stack([mu1, mu1])
    omega = np.full((H, K, d), -30.0)
    alpha = np.zeros((H, K))
    lab = np.array([0] * 12 + [1] * 6 + [2] * 6)           # component 3 unused
    r.shuffle(lab)
    Qx = np.stack([mu1[lab], mu1[lab]])[None]
    p, husage, htoken, rmax, z = oracle.diagnostics(Qx, mu, omega, alpha, 1e-4)
    freq = np.bincount(lab, minlength=K) / N
    np.testing.assert_allclose(p, freq, atol=1e-12)
    assert husage == pytest.approx(-(0.5 * np.log(0.5) + 2 * 0.25 * np.log(0.25)) / np.log(K), rel=1e-12)
    assert htoken == pytest.approx(0.0, abs=1e-12)
    assert rmax == pytest.approx(1.0, abs=1e-12)
    assert np.array_equal(z[0], lab)


def test_diagnostics_invariants_and_head_symmetry():
    x = make_heads(B=3, H=4, N=20, K=7, seed=11)
    K = 7
    p, husage, htoken, rmax, z = oracle.diagnostics(x["Qx"], x["mu"], x["omega"], x["alpha"], 1e-4)
    assert p.sum() == pytest.approx(1.0, rel=1e-12) and (p > 0).all()
    # Jensen: the entropy of the mean is at least the mean entropy
    assert 0.0 <= htoken <= husage <= 1.0
    assert 1.0 / K <= rmax <= 1.0
    assert z.min() >= 0 and z.max() < K
    # the head average does not depend on the order of the heads
    perm = np.array([2, 0, 3, 1])
    y = oracle.diagnostics(x["Qx"][:, perm], x["mu"][perm], x["omega"][perm], x["alpha"][perm], 1e-4)
    np.testing.assert_allclose(y[0], p, rtol=1e-12)
    assert y[1:4] == pytest.approx((husage, htoken, rmax), rel=1e-12)
    assert np.array_equal(y[4], z)
    # H copies of one head give that head's own diagnostics
    one = {k: v[:, :1] if k == "Qx" else v[:1] for k, v in x.items()}
    rep = {k: np.repeat(v, 3, axis=1 if k == "Qx" else 0) for k, v in one.items()}
    a = oracle.diagnostics(one["Qx"], one["mu"], one["omega"], one["alpha"], 1e-4)
    b = oracle.diagnostics(rep["Qx"], rep["mu"], rep["omega"], rep["alpha"], 1e-4)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12)
    assert a[1:4] == pytest.approx(b[1:4], rel=1e-12)


# ---------------------------------------------------------------- cross-attention (sections 3.1, 6)

def brute_force_cross(Qx, Ky, Vy, mu, omega, alpha, var_floor, eps):
    """Explicit Nq x Nkv affinity Gamma^Q_X Gamma^K_Y^T, row-normalised, applied to Vy."""
    At = textbook_gamma(Qx, mu, omega, alpha, var_floor) @ textbook_gamma(Ky, mu, omega, alpha, var_floor).T
    return (At / (At.sum(axis=1, keepdims=True) + eps)) @ Vy


@pytest.mark.parametrize("Nq,Nkv,eps", [(17, 40, 1e-6), (50, 3, 0.2), (1, 1, 1e-6), (9, 9, 0.05)])
def test_cross_matches_explicit_affinity(Nq, Nkv, eps):
    r = np.random.default_rng(Nq * 100 + Nkv)
    d, K, dv = 4, 6, 5
    Qx, Ky, Vy = r.normal(size=(Nq, d)), r.normal(size=(Nkv, d)), r.normal(size=(Nkv, dv))
    mu, omega, alpha = r.normal(size=(K, d)), 0.5 * r.normal(size=(K, d)), r.normal(size=(K,))
    got = oracle.cross_head(Qx, Ky, Vy, mu, omega, alpha, 1e-4, eps)
    np.testing.assert_allclose(got, brute_force_cross(Qx, Ky, Vy, mu, omega, alpha, 1e-4, eps), rtol=1e-9,
                               atol=1e-12)


def test_cross_with_the_sequence_itself_is_self_attention():
    x = make(N=33)
    got = oracle.cross_head(x["Qx"], x["Kx"], x["V"], x["mu"], x["omega"], x["alpha"], 1e-4, 1e-6)
    ref = oracle.forward_head(x["Qx"], x["Kx"], x["V"], x["mu"], x["omega"], x["alpha"], 1e-4, 1e-6, False)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_cross_context_order_does_not_matter_and_queries_are_independent():
    r = np.random.default_rng(5)
    d, K, dv, Nq, Nkv = 3, 4, 2, 12, 30
    Qx, Ky, Vy = r.normal(size=(Nq, d)), r.normal(size=(Nkv, d)), r.normal(size=(Nkv, dv))
    mu, omega, alpha = r.normal(size=(K, d)), 0.5 * r.normal(size=(K, d)), r.normal(size=(K,))
    base = oracle.cross_head(Qx, Ky, Vy, mu, omega, alpha, 1e-4, 1e-6)
    perm = r.permutation(Nkv)
    np.testing.assert_allclose(oracle.cross_head(Qx, Ky[perm], Vy[perm], mu, omega, alpha, 1e-4, 1e-6), base,
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.cross_head(Qx[:5], Ky, Vy, mu, omega, alpha, 1e-4, 1e-6), base[:5],
                               rtol=1e-12, atol=1e-14)


# ---- backward pass (section 4.1, Eqs. 17-20; Eqs. 14-15 for the reparameterised parameters) ----

BWD_INPUTS = ("Qx", "Kx", "V", "mu", "omega", "alpha")


def loss_brute_force(x, dO, var_floor, eps, causal):
    """L = sum(dO * O) with O from the explicit affinity of Eq. (9)-(10) / (9b)-(10b)
    and scipy's densities: shares no code with the oracle."""
    O, _, _ = brute_force(x["Qx"], x["Kx"], x["V"], x["mu"], x["omega"], x["alpha"], var_floor, eps, causal)
    return float((dO * O).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences_of_the_explicit_affinity(causal):
    # every input entry perturbed in turn; eps large enough that its placement matters
    var_floor, eps, h = 1e-3, 0.1, 1e-5
    x = make(N=6, d=2, K=3, dv=2, seed=21 + causal)
    dO = np.random.default_rng(5).normal(size=(6, 2))
    g = oracle.backward_head(x["Qx"], x["Kx"], x["V"], x["mu"], x["omega"], x["alpha"], var_floor, eps,
                             causal, dO)
    for name in BWD_INPUTS:
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            xp = {k: v.copy() for k, v in x.items()}
            xm = {k: v.copy() for k, v in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (loss_brute_force(xp, dO, var_floor, eps, causal) -
                       loss_brute_force(xm, dO, var_floor, eps, causal)) / (2 * h)
        scale = max(np.abs(fd).max(), 1e-3)
        assert np.abs(g[name] - fd).max() <= 1e-6 * scale, (name, g[name], fd)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_directional_derivative_on_a_larger_head(causal):
    # all inputs moved along one random direction at once, at K = 9, N = 60
    var_floor, eps, h = 1e-4, 1e-3, 1e-6
    x = make(N=60, d=6, K=9, dv=5, seed=30 + causal)
    r = np.random.default_rng(31)
    dO = r.normal(size=(60, 5))
    delta = {k: r.normal(size=v.shape) for k, v in x.items()}
    g = oracle.backward_head(*(x[k] for k in BWD_INPUTS), var_floor, eps, causal, dO)

    def loss(s):
        y = {k: x[k] + s * delta[k] for k in x}
        return float((dO * oracle.forward_head(*(y[k] for k in BWD_INPUTS), var_floor, eps, causal)).sum())

    fd = (loss(h) - loss(-h)) / (2 * h)
    an = sum(float((g[k] * delta[k]).sum()) for k in BWD_INPUTS)
    assert abs(fd - an) <= 1e-6 * max(abs(an), 1.0), (fd, an)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    var_floor, eps = 1e-4, 1e-3
    x = make(N=50, d=4, K=6, dv=3, seed=40 + causal)
    dO = np.random.default_rng(41).normal(size=(50, 3))
    g = oracle.backward_head(*(x[k] for k in BWD_INPUTS), var_floor, eps, causal, dO)
    O = oracle.forward_head(*(x[k] for k in BWD_INPUTS), var_floor, eps, causal)
    # a common shift of every routing vector and every mean leaves each score unchanged
    shift = g["Qx"].sum(axis=0) + g["Kx"].sum(axis=0) + g["mu"].sum(axis=0)
    assert np.abs(shift).max() <= 1e-10 * max(np.abs(g["mu"]).max(), 1.0)
    # O is homogeneous of degree one in V (Eq. 7-8): Euler's identity
    assert abs((g["V"] * x["V"]).sum() - (dO * O).sum()) <= 1e-10 * np.abs(dO * O).sum()
    # the priors enter through log_softmax(alpha) (Eq. 15): a common shift of alpha does nothing
    assert abs(g["alpha"].sum()) <= 1e-12 * max(np.abs(g["alpha"]).max(), 1.0)


def test_causal_backward_reaches_only_the_prefix():
    # dO nonzero at row t only: queries other than t get nothing, keys and values after t nothing
    var_floor, eps, t = 1e-4, 1e-3, 23
    x = make(N=40, d=4, K=5, dv=3, seed=50)
    dO = np.zeros((40, 3))
    dO[t] = np.random.default_rng(51).normal(size=3)
    g = oracle.backward_head(*(x[k] for k in BWD_INPUTS), var_floor, eps, True, dO)
    others = np.arange(40) != t
    assert np.abs(g["Qx"][others]).max() == 0.0 and np.abs(g["Qx"][t]).max() > 0
    assert np.abs(g["Kx"][t + 1:]).max() == 0.0 and np.abs(g["V"][t + 1:]).max() == 0.0
    assert np.abs(g["Kx"][:t + 1]).max() > 0 and np.abs(g["V"][:t + 1]).max() > 0


# ---- input projections (section 3.1, Eq. 4)

def test_project_matches_brute_force_and_a_library_matmul():
    # pure-Python triple loop on a tiny case, and numpy's einsum on a larger one
    rng = np.random.default_rng(60)
    B, N, D, H, d, dv = 2, 3, 5, 2, 2, 3
    X, Wq, Wk, Wv = (rng.normal(size=s) for s in ((B, N, D), (H, D, d), (H, D, d), (H, D, dv)))
    Qx, Kx, V = oracle.project(X, Wq, Wk, Wv)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                for c in range(d):
                    assert abs(Qx[b, h, i, c] - sum(X[b, i, m] * Wq[h, m, c] for m in range(D))) <= 1e-12
                    assert abs(Kx[b, h, i, c] - sum(X[b, i, m] * Wk[h, m, c] for m in range(D))) <= 1e-12
                for c in range(dv):
                    assert abs(V[b, h, i, c] - sum(X[b, i, m] * Wv[h, m, c] for m in range(D))) <= 1e-12
    B, N, D, H, d, dv = 2, 40, 96, 3, 8, 16
    X, Wq, Wk, Wv = (rng.normal(size=s) for s in ((B, N, D), (H, D, d), (H, D, d), (H, D, dv)))
    Qx, Kx, V = oracle.project(X, Wq, Wk, Wv)
    for got, W in ((Qx, Wq), (Kx, Wk), (V, Wv)):
        assert np.abs(got - np.einsum("bnm,hmc->bhnc", X, W)).max() <= 1e-12


def test_project_with_unit_columns_selects_input_features():
    # W with a single 1 per column picks features of X: head h's Qx column c is X[:, :, c + h]
    rng = np.random.default_rng(61)
    B, N, D, H, d = 1, 7, 6, 2, 3
    X = rng.normal(size=(B, N, D))
    Wq = np.zeros((H, D, d))
    for h in range(H):
        for c in range(d):
            Wq[h, c + h, c] = 1.0
    Qx, Kx, V = oracle.project(X, Wq, 2 * Wq, -Wq)
    for h in range(H):
        assert np.array_equal(Qx[0, h], X[0][:, h:h + d])
        assert np.array_equal(Kx[0, h], 2 * X[0][:, h:h + d])
        assert np.array_equal(V[0, h], -X[0][:, h:h + d])
