"""Pins for the fp64 oracle: checks against what the GMA page and mathematics fix, never against
the oracle itself or the CUDA library.

Page: "Attention par Mélange Gaussien (GMA)", gist.science/fr/paper/2606.18283, Méthodologie
§1 (posterior responsibilities), §2 (write / read phases, O = Gamma_Q V~ / (Gamma_Q Z + eps),
implicit affinity A~ = Gamma_Q Gamma_K^T), §3 (causal prefix sums; softplus variances, softmax
priors), Contributions §3 (affinity is non-negative with rank <= K).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import norm

import oracle
from oracle import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, B=2, H=2, N=37, d_r=5, K=7, d_v=3, mu_std=1.0):
    r = np.random.default_rng(seed)
    return dict(
        QX=r.standard_normal((B, H, N, d_r)),
        KX=r.standard_normal((B, H, N, d_r)),
        V=r.standard_normal((B, H, N, d_v)),
        mu=r.standard_normal((H, K, d_r)) * mu_std,
        raw=r.standard_normal((H, K, d_r)) * 0.5,
        logits=r.standard_normal((H, K)),
    )


def _fwd(c, causal, floor=1e-3, eps=1e-6, **over):
    d = dict(c)
    d.update(over)
    return oracle.forward(causal, d["QX"], d["KX"], d["V"], d["mu"], d["raw"], d["logits"],
                          floor, eps)


# ---------------------------------------------------------------- reparametrisation (§3)

def test_softplus_variance_closed_forms():
    raw = np.array([[0.0, math.log(math.e - 1.0), 40.0, -40.0, -800.0, 700.0]])
    var, _ = oracle.params(raw, np.zeros(1), 0.0)
    expect = [math.log(2.0), 1.0, 40.0 + math.log1p(math.exp(-40.0)), math.exp(-40.0),
              0.0, 700.0]
    np.testing.assert_allclose(var[0, :4], expect[:4], rtol=1e-14)
    assert var[0, 4] >= 0.0 and var[0, 4] < 1e-300
    assert var[0, 5] == 700.0
    var_f, _ = oracle.params(raw, np.zeros(1), 1e-3)
    np.testing.assert_allclose(var_f - var, 1e-3, atol=1e-12)


def test_prior_logits_are_log_softmax():
    logits = np.array([0.3, -1.2, 2.5, 0.0, 7.0])
    _, logpi = oracle.params(np.zeros((5, 1)), logits, 0.0)
    np.testing.assert_allclose(np.exp(logpi), softmax(logits), rtol=1e-14)
    np.testing.assert_allclose(np.exp(logpi).sum(), 1.0, rtol=1e-15)
    _, logpi_shift = oracle.params(np.zeros((5, 1)), logits + 123.0, 0.0)
    np.testing.assert_allclose(logpi_shift, logpi, atol=1e-12)


# ---------------------------------------------------------------- posterior (§1)

def test_P1_responsibilities_nonnegative_rows_sum_to_one():
    c = _rand_case(0, N=200, d_r=16, K=32)
    g = oracle.responsibilities(c["QX"][0, 0], c["mu"][0], c["raw"][0], c["logits"][0], 1e-3)
    assert (g >= 0).all()
    np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-14)


def test_P7_posterior_matches_scipy_normal_logpdf_and_softmax():
    c = _rand_case(1, N=64, d_r=9, K=11, mu_std=1.5)
    X, mu, raw, lg = c["QX"][0, 1], c["mu"][1], c["raw"][1], c["logits"][1]
    g = oracle.responsibilities(X, mu, raw, lg, 1e-3)
    var = np.logaddexp(0.0, raw) + 1e-3
    logp = norm.logpdf(X[:, None, :], loc=mu[None], scale=np.sqrt(var)[None]).sum(-1)
    expect = softmax(logp + np.log(softmax(lg))[None], axis=1)
    np.testing.assert_allclose(g, expect, rtol=1e-12, atol=1e-15)


def test_P10_translation_invariance():
    c = _rand_case(2, N=50, d_r=6, K=5)
    X, mu, raw, lg = c["QX"][0, 0], c["mu"][0], c["raw"][0], c["logits"][0]
    t = np.array([0.7, -1.3, 2.0, 0.1, -0.4, 3.0])
    g0 = oracle.responsibilities(X, mu, raw, lg, 1e-3)
    g1 = oracle.responsibilities(X + t, mu + t, raw, lg, 1e-3)
    np.testing.assert_allclose(g1, g0, rtol=1e-11, atol=1e-14)


def test_P11_identical_components_uniform_prior_give_one_over_K():
    K, d_r = 6, 4
    mu = np.tile(np.array([[0.3, -0.2, 1.0, 0.5]]), (K, 1))
    raw = np.tile(np.array([[0.1, -0.5, 0.9, 0.0]]), (K, 1))
    X = np.random.default_rng(3).standard_normal((20, d_r))
    g = oracle.responsibilities(X, mu, raw, np.zeros(K), 1e-3)
    np.testing.assert_allclose(g, 1.0 / K, rtol=1e-14)


def test_golden_two_component_logistic():
    fx = json.load(open(os.path.join(GOLDEN, "two_component_logistic.json")))
    g = oracle.responsibilities(np.array(fx["QX"]), np.array(fx["mu"]), np.array(fx["raw"]),
                                np.array(fx["logits"]), fx["var_floor"])
    np.testing.assert_allclose(g, fx["gamma"], rtol=1e-13)
    for causal, key in ((False, "bidir"), (True, "causal")):
        O = oracle.forward(causal, np.array(fx["QX"])[None, None], np.array(fx["KX"])[None, None],
                           np.array(fx["V"])[None, None], np.array(fx["mu"])[None],
                           np.array(fx["raw"])[None], np.array(fx["logits"])[None],
                           fx["var_floor"], fx["eps"])
        num = np.array(fx[key + "_num"])
        den = np.array(fx[key + "_den"])
        np.testing.assert_allclose(O[0, 0, :, 0], num / (den + fx["eps"]), rtol=1e-13)


def test_golden_equal_means_unequal_variance_log_determinant():
    fx = json.load(open(os.path.join(GOLDEN, "equal_means_unequal_variance.json")))
    mu, raw, lg = np.array(fx["mu"]), np.array(fx["raw"]), np.array(fx["logits"])
    g = oracle.responsibilities(np.array(fx["X_rational"]), mu, raw, lg, fx["var_floor"])
    np.testing.assert_allclose(g, fx["gamma_rational"], rtol=1e-13)
    x_tie = math.sqrt(8.0 * math.log(2.0) / 3.0)
    x = np.array([[x_tie], [2.0]])
    g = oracle.responsibilities(x, mu, raw, lg, fx["var_floor"])
    np.testing.assert_allclose(g[0], [0.5, 0.5], rtol=1e-13)
    g1 = 2.0 / (2.0 + math.exp(1.5))
    np.testing.assert_allclose(g[1], [g1, 1.0 - g1], rtol=1e-13)


# ---------------------------------------------------------------- write / read (§2, §3)

@pytest.mark.parametrize("causal", [False, True])
def test_P2_linear_form_equals_explicit_affinity(causal):
    c = _rand_case(4)
    O1 = _fwd(c, causal)
    O2 = bruteforce.forward(causal, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"],
                            1e-3, 1e-6)
    np.testing.assert_allclose(O1, O2, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_P2_linear_form_equals_explicit_affinity_wide(causal):
    c = _rand_case(5, B=1, H=1, N=256, d_r=16, K=8, d_v=32)
    O1 = _fwd(c, causal)
    O2 = bruteforce.forward(causal, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"],
                            1e-3, 1e-6)
    np.testing.assert_allclose(O1, O2, rtol=1e-11, atol=1e-13)


def test_P3_P4_affinity_nonnegative_rank_at_most_K():
    c = _rand_case(6, N=60, d_r=4, K=5)
    A = bruteforce.affinity(c["QX"][0, 0], c["KX"][0, 0], c["mu"][0], c["raw"][0],
                            c["logits"][0], 1e-3)
    assert (A >= 0).all()
    s = np.linalg.svd(A, compute_uv=False)
    assert s[5] / s[0] <= 1e-12
    assert s[4] / s[0] > 1e-8   # generic case: exactly rank K


@pytest.mark.parametrize("causal", [False, True])
def test_P5_single_component_gives_mean_or_running_mean(causal):
    c = _rand_case(7, K=1)
    eps = 1e-6
    O = _fwd(c, causal, eps=eps)
    V = c["V"]
    N = V.shape[2]
    if causal:
        expect = np.cumsum(V, axis=2) / (np.arange(1, N + 1)[None, None, :, None] + eps)
    else:
        expect = V.sum(axis=2, keepdims=True) / (N + eps) * np.ones_like(V)
    np.testing.assert_allclose(O, expect, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_P6_constant_values_are_reproduced(causal):
    c = _rand_case(8)
    V = np.full_like(c["V"], -2.75)
    O = _fwd(c, causal, eps=0.0, V=V)
    np.testing.assert_allclose(O, -2.75, rtol=1e-13)
    # with eps > 0 the first causal row is scaled by den/(den+eps), den = gamma_Q0 . gamma_K0
    eps = 0.05
    O = _fwd(c, causal, eps=eps, V=V)
    if causal:
        gq = oracle.responsibilities(c["QX"][0, 0, :1], c["mu"][0], c["raw"][0], c["logits"][0],
                                     1e-3)
        gk = oracle.responsibilities(c["KX"][0, 0, :1], c["mu"][0], c["raw"][0], c["logits"][0],
                                     1e-3)
        den = float(gq[0] @ gk[0])
        np.testing.assert_allclose(O[0, 0, 0], -2.75 * den / (den + eps), rtol=1e-12)
    assert (np.abs(O) <= 2.75 * (1 + 1e-12)).all()


def test_P8_causal_last_row_equals_bidirectional_last_row():
    c = _rand_case(9)
    Ob = _fwd(c, False)
    Oc = _fwd(c, True)
    np.testing.assert_allclose(Oc[:, :, -1], Ob[:, :, -1], rtol=1e-12)
    assert np.abs(Oc[:, :, 0] - Ob[:, :, 0]).max() > 1e-3


def test_P9_component_permutation_and_row_symmetries():
    c = _rand_case(10)
    perm = np.random.default_rng(0).permutation(c["mu"].shape[1])
    for causal in (False, True):
        O = _fwd(c, causal)
        Op = _fwd(c, causal, mu=c["mu"][:, perm], raw=c["raw"][:, perm],
                  logits=c["logits"][:, perm])
        np.testing.assert_allclose(Op, O, rtol=1e-12, atol=1e-14)
    O = _fwd(c, False)
    rp = np.random.default_rng(1).permutation(c["KX"].shape[2])
    Ok = _fwd(c, False, KX=c["KX"][:, :, rp], V=c["V"][:, :, rp])
    np.testing.assert_allclose(Ok, O, rtol=1e-12, atol=1e-14)
    Oq = _fwd(c, False, QX=c["QX"][:, :, rp])
    np.testing.assert_allclose(Oq, O[:, :, rp], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_P12_output_is_linear_in_values(causal):
    c = _rand_case(11)
    V2 = np.random.default_rng(12).standard_normal(c["V"].shape)
    O1 = _fwd(c, causal)
    O2 = _fwd(c, causal, V=V2)
    O3 = _fwd(c, causal, V=2.5 * c["V"] - 0.5 * V2)
    np.testing.assert_allclose(O3, 2.5 * O1 - 0.5 * O2, rtol=1e-11, atol=1e-12)


def test_P13_hard_clusters_give_group_means():
    # three far-apart tight components; each token sits on one of them -> one-hot gammas
    K, d_r, N, d_v = 3, 2, 30, 4
    centres = np.array([[0.0, 0.0], [50.0, 0.0], [0.0, 50.0]])
    lab = np.random.default_rng(13).integers(0, K, N)
    X = centres[lab] + 0.01 * np.random.default_rng(14).standard_normal((N, d_r))
    V = np.random.default_rng(15).standard_normal((N, d_v))
    raw = np.full((K, d_r), -3.0)
    args = (X[None, None], X[None, None], V[None, None], centres[None], raw[None],
            np.zeros((1, K)), 1e-3, 0.0)
    g = oracle.responsibilities(X, centres, raw, np.zeros(K), 1e-3)
    assert np.abs(g - np.eye(K)[lab]).max() < 1e-12
    Ob = oracle.forward(False, *args)[0, 0]
    Oc = oracle.forward(True, *args)[0, 0]
    for i in range(N):
        same = lab == lab[i]
        np.testing.assert_allclose(Ob[i], V[same].mean(0), rtol=1e-10, atol=1e-12)
        prev = same & (np.arange(N) <= i)
        np.testing.assert_allclose(Oc[i], V[prev].mean(0), rtol=1e-10, atol=1e-12)


def test_oracle_threads_do_not_change_results():
    c = _rand_case(16, B=3, H=2, N=40)
    O1, used1 = oracle.forward(True, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"],
                               1e-3, 1e-6, nthreads=1, return_threads=True)
    O4 = oracle.forward(True, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3,
                        1e-6, nthreads=4)
    assert used1 == 1
    np.testing.assert_array_equal(O1, O4)


# ---------------------------------------------------------------- planted mistakes

def _mutant_posterior(X, mu, var, logpi, drop_logdet=False, flip_mean=False):
    m = -mu if flip_mean else mu
    q = ((X[:, None, :] - m[None]) ** 2 / var[None]).sum(-1)
    if not drop_logdet:
        q = q + np.log(var).sum(-1)[None]
    return softmax(logpi[None] - 0.5 * q, axis=1)


def test_pins_catch_planted_mistakes():
    """Each plausible slip, planted in a CPU restatement, moves the result well past the pins'
    tolerances, so the pins above would reject an oracle that made it."""
    c = _rand_case(17, N=40, d_r=5, K=6)
    X, mu, raw, lg = c["QX"][0, 0], c["mu"][0], c["raw"][0], c["logits"][0]
    var, logpi = oracle.params(raw, lg, 1e-3)
    good = oracle.responsibilities(X, mu, raw, lg, 1e-3)
    ok = _mutant_posterior(X, mu, var, logpi)
    np.testing.assert_allclose(ok, good, rtol=1e-12, atol=1e-15)
    for kw in ({"drop_logdet": True}, {"flip_mean": True}):
        assert np.abs(_mutant_posterior(X, mu, var, logpi, **kw) - good).max() > 1e-3
    # transposed affinity and exclusive prefix both break P2
    A = bruteforce.affinity(X, c["KX"][0, 0], mu, raw, lg, 1e-3)
    V = c["V"][0, 0]
    O = _fwd(c, True)[0, 0]
    At = np.tril(A.T)
    assert np.abs(At @ V / (At.sum(1, keepdims=True) + 1e-6) - O).max() > 1e-3
    Ae = np.tril(A, -1)
    assert np.abs(Ae @ V / (Ae.sum(1, keepdims=True) + 1e-6) - O).max() > 1e-3


# ---------------------------------------------------------------- decode step and cross-attention

def test_decode_steps_reproduce_the_causal_affinity_form():
    """N decode steps from an empty memory give the causal rows of the explicit affinity form
    (Méthodologie §3), and the final memory is sum_j gamma_K,j [v_j, 1] by scipy's posterior."""
    c = _rand_case(11, N=13)
    B, H, N, d_r = c["QX"].shape
    d_v = c["V"].shape[-1]
    K = c["mu"].shape[1]
    S = np.zeros((B, H, K, d_v + 1))
    outs = []
    for i in range(N):
        o, S = oracle.decode_step(c["QX"][:, :, i], c["KX"][:, :, i], c["V"][:, :, i], c["mu"],
                                  c["raw"], c["logits"], 1e-3, 1e-6, S)
        outs.append(o)
    got = np.stack(outs, axis=2)
    ref = bruteforce.forward(True, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3, 1e-6)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    for b in range(B):
        for h in range(H):
            var = bruteforce.softplus(c["raw"][h]) + 1e-3
            g = bruteforce.posterior(c["KX"][b, h], c["mu"][h], var, c["logits"][h])
            mem = g.T @ np.concatenate([c["V"][b, h], np.ones((N, 1))], axis=1)
            np.testing.assert_allclose(S[b, h], mem, rtol=1e-12, atol=1e-12)


def test_decode_step_leaves_the_input_state_alone_and_adds_one_token():
    c = _rand_case(12, N=1)
    B, H, _, d_r = c["QX"].shape
    K = c["mu"].shape[1]
    d_v = c["V"].shape[-1]
    S0 = np.random.default_rng(3).random((B, H, K, d_v + 1))
    keep = S0.copy()
    o, S1 = oracle.decode_step(c["QX"][:, :, 0], c["KX"][:, :, 0], c["V"][:, :, 0], c["mu"],
                               c["raw"], c["logits"], 1e-3, 0.0, S0)
    assert np.array_equal(S0, keep)
    for b in range(B):
        for h in range(H):
            var = bruteforce.softplus(c["raw"][h]) + 1e-3
            gk = bruteforce.posterior(c["KX"][b, h], c["mu"][h], var, c["logits"][h])[0]
            gq = bruteforce.posterior(c["QX"][b, h], c["mu"][h], var, c["logits"][h])[0]
            add = np.outer(gk, np.append(c["V"][b, h, 0], 1.0))
            np.testing.assert_allclose(S1[b, h] - S0[b, h], add, atol=1e-12)
            np.testing.assert_allclose(o[b, h], gq @ S1[b, h][:, :d_v] / (gq @ S1[b, h][:, d_v]),
                                       rtol=1e-12)


@pytest.mark.parametrize("nq,nk", [(5, 23), (31, 4), (1, 1)])
def test_cross_attention_equals_explicit_affinity(nq, nk):
    """Nq queries reading the memory of Nk keys (the bidirectional path with N_q != N_k) equals
    A~ V / (A~ 1 + eps) with the rectangular A~ = Gamma_Q Gamma_K^T."""
    r = np.random.default_rng(nq * 100 + nk)
    B, H, d_r, K, d_v = 2, 2, 5, 6, 3
    QX = r.standard_normal((B, H, nq, d_r))
    KX = r.standard_normal((B, H, nk, d_r))
    V = r.standard_normal((B, H, nk, d_v))
    mu = r.standard_normal((H, K, d_r))
    raw = r.standard_normal((H, K, d_r)) * 0.5
    logits = r.standard_normal((H, K))
    got = oracle.forward_cross(QX, KX, V, mu, raw, logits, 1e-3, 1e-6)
    for b in range(B):
        for h in range(H):
            ref = bruteforce.forward_slice(False, QX[b, h], KX[b, h], V[b, h], mu[h], raw[h], logits[h],
                                   1e-3, 1e-6)
            np.testing.assert_allclose(got[b, h], ref, rtol=0, atol=1e-12)


def test_cross_attention_row_symmetries():
    """The read sums over keys (Methodologie §2: V~ = Gamma_K^T V, Z = Gamma_K^T 1), so permuting
    the key rows jointly with their value rows leaves O unchanged, permuting the query rows
    permutes the output rows the same way, and appending a key whose value row is zero only adds
    its responsibilities to the normaliser (O shrinks row by row, never changes sign)."""
    r = np.random.default_rng(41)
    B, H, nq, nk, d_r, K, d_v = 2, 2, 7, 11, 4, 5, 3
    QX = r.standard_normal((B, H, nq, d_r))
    KX = r.standard_normal((B, H, nk, d_r))
    V = r.standard_normal((B, H, nk, d_v))
    mu = r.standard_normal((H, K, d_r))
    raw = r.standard_normal((H, K, d_r)) * 0.5
    logits = r.standard_normal((H, K))
    base = oracle.forward_cross(QX, KX, V, mu, raw, logits, 1e-3, 1e-6)
    pk = r.permutation(nk)
    got = oracle.forward_cross(QX, KX[:, :, pk], V[:, :, pk], mu, raw, logits, 1e-3, 1e-6)
    np.testing.assert_allclose(got, base, rtol=0, atol=1e-13)
    pq = r.permutation(nq)
    got = oracle.forward_cross(QX[:, :, pq], KX, V, mu, raw, logits, 1e-3, 1e-6)
    np.testing.assert_allclose(got, base[:, :, pq], rtol=0, atol=1e-13)
    KX2 = np.concatenate([KX, r.standard_normal((B, H, 1, d_r))], axis=2)
    V2 = np.concatenate([V, np.zeros((B, H, 1, d_v))], axis=2)
    got = oracle.forward_cross(QX, KX2, V2, mu, raw, logits, 1e-3, 1e-6)
    ratio = got / base
    assert np.all(ratio > 0) and np.all(ratio < 1)
    # the shrink factor is one number per query row: the same for every value column
    np.testing.assert_allclose(ratio, np.broadcast_to(ratio[..., :1], ratio.shape), rtol=1e-10)


def test_cross_attention_with_equal_lengths_is_the_bidirectional_forward():
    c = _rand_case(13, N=17)
    got = oracle.forward_cross(c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3, 1e-6)
    np.testing.assert_allclose(got, _fwd(c, False), rtol=0, atol=1e-13)


# ------------------------------------------------------------------ usage diagnostics
def test_usage_histogram_closed_forms():
    """Hand-countable assignments: counts, used components and the normalised entropy."""
    K = 4
    a = np.array([[[0, 0, 1, 1], [3, 3, 3, 3]]])            # B=1, H=2, N=4
    counts, used, ent = oracle.usage_from_assign(a, K)
    assert counts.tolist() == [[2, 2, 0, 0], [0, 0, 0, 4]]
    assert used.tolist() == [2, 1]
    assert ent[0] == pytest.approx(np.log(2) / np.log(4), abs=1e-15)   # two equal halves: 1/2
    assert ent[1] == 0.0                                                # one component: 0
    uniform = np.arange(8 * K).reshape(1, 1, -1) % K
    _, used_u, ent_u = oracle.usage_from_assign(uniform, K)
    assert used_u[0] == K and ent_u[0] == pytest.approx(1.0, abs=1e-15)
    _, _, ent_1 = oracle.usage_from_assign(np.zeros((2, 1, 3), dtype=int), 1)
    assert ent_1[0] == 0.0


def test_usage_of_hard_clusters_recovers_the_clusters():
    """Well-separated components, tokens drawn near one mean each: the hard assignment is the
    cluster, the mass is the cluster size (responsibilities ~ one-hot)."""
    rng = np.random.default_rng(5)
    K, d_r = 3, 4
    mu = np.array([[0.0] * d_r, [12.0] * d_r, [-12.0] * d_r])[None]
    raw = np.full((1, K, d_r), -2.0)      # small variances
    logits = np.zeros((1, K))
    labels = np.array([0, 1, 2, 2, 1, 0, 0, 2, 1, 1])
    X = (mu[0][labels] + 0.05 * rng.standard_normal((labels.size, d_r)))[None, None]
    u = oracle.usage(X, mu, raw, logits, 1e-3)
    assert u["assign"][0, 0].tolist() == labels.tolist()
    assert u["counts"][0].tolist() == np.bincount(labels, minlength=K).tolist()
    assert np.allclose(u["mass"][0], np.bincount(labels, minlength=K), atol=1e-9)
    assert np.allclose(u["gamma_max"], 1.0, atol=1e-9)


def test_usage_invariants_and_component_permutation():
    """Counts and masses sum to the token count; assignments are the argmax of the oracle's
    posterior; permuting the components permutes counts and masses."""
    c = _rand_case(11, B=2, H=3, N=41, d_r=5, K=6)
    u = oracle.usage(c["QX"], c["mu"], c["raw"], c["logits"], 1e-3)
    assert (u["counts"].sum(axis=1) == 2 * 41).all()
    assert np.allclose(u["mass"].sum(axis=1), 2 * 41, rtol=1e-12)
    assert ((u["used"] >= 1) & (u["used"] <= 6)).all()
    assert ((u["entropy"] >= 0) & (u["entropy"] <= 1)).all()
    for b, h in [(0, 0), (1, 2)]:
        var = bruteforce.softplus(c["raw"][h]) + 1e-3
        g = bruteforce.posterior(c["QX"][b, h], c["mu"][h], var, c["logits"][h])
        assert (np.argmax(g, axis=1) == u["assign"][b, h]).all()
        assert np.allclose(g.max(axis=1), u["gamma_max"][b, h], rtol=1e-12)
    perm = np.array([3, 0, 5, 1, 4, 2])
    up = oracle.usage(c["QX"], c["mu"][:, perm], c["raw"][:, perm], c["logits"][:, perm], 1e-3)
    assert (up["counts"] == u["counts"][:, perm]).all()
    assert np.allclose(up["mass"], u["mass"][:, perm], rtol=1e-12)
    assert np.allclose(up["entropy"], u["entropy"], rtol=1e-12)


# ------------------------------------------------------------------ backward pass
def _loss(causal, c, dO, floor=1e-3, eps=1e-6):
    return float((_fwd(c, causal, floor, eps) * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(causal):
    """Every gradient of sum(dO * O) against central differences of the forward oracle (fp64,
    step 1e-6): a dropped term, a wrong sign or a transposed operand anywhere fails this."""
    c = _rand_case(21, B=2, H=2, N=6, d_r=3, K=4, d_v=2)
    rng = np.random.default_rng(22)
    dO = rng.standard_normal((2, 2, 6, 2))
    grads = oracle.backward(causal, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3,
                            1e-6, dO)
    names = ["QX", "KX", "V", "mu", "raw", "logits"]
    h = 1e-6
    for name, g in zip(names, grads):
        base = c[name]
        flat = base.reshape(-1)
        num = np.empty(flat.size)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(causal, c, dO)
            flat[i] = old - h
            lm = _loss(causal, c, dO)
            flat[i] = old
            num[i] = (lp - lm) / (2 * h)
        scale = max(np.abs(num).max(), 1e-3)
        assert np.abs(g.reshape(-1) - num).max() <= 1e-6 * scale + 1e-8, name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    """Translation x -> x + t, mu -> mu + t leaves the output unchanged, so the gradients of the
    routing rows and of the means sum to zero per head and dimension; the prior gradient sums to
    zero over the components (log softmax); dV is linear in dO."""
    c = _rand_case(23, B=2, H=2, N=9, d_r=4, K=5, d_v=3)
    dO = np.random.default_rng(24).standard_normal((2, 2, 9, 3))
    g = oracle.backward(causal, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3, 1e-6, dO)
    dQX, dKX, dV, dmu, draw, dlog = g
    tot = dQX.sum(axis=(0, 2)) + dKX.sum(axis=(0, 2)) + dmu.sum(axis=1)
    assert np.abs(tot).max() <= 1e-10 * max(1.0, np.abs(dmu).max())
    assert np.abs(dlog.sum(axis=1)).max() <= 1e-12 * max(1.0, np.abs(dlog).max())
    g2 = oracle.backward(causal, c["QX"], c["KX"], c["V"], c["mu"], c["raw"], c["logits"], 1e-3, 1e-6, 2.5 * dO)
    assert np.allclose(g2[2], 2.5 * dV, rtol=1e-12, atol=1e-14)
