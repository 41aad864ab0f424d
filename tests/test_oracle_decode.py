"""Pins of the fp64 oracle's decode step against facts fixed outside it:
closed forms, identities the pages state, brute force and numpy routines.

Sources: MomentKV (arXiv 2606.01563) sec 2, 4.1-4.2, Algorithm 1, App. A-C;
InertiaKV (arXiv 2609.03515) sec 3.1 eqs 1-4; KeepKV reading notes (arXiv
2504.09936) eqs 1-3, 6, 23.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import oracle as O


def bf(x):
    return O.bf16_round(x)


def make_session(k, v, vote=None, G=None, cap=None):
    """One-unit session from float arrays (bf16-exact)."""
    k = np.asarray(k, float)
    n, d = k.shape
    s = O.DecodeSession(1, 1 if G is None else G, d, cap or n + 4)
    s.load(0, k, v, vote)
    return s


# ---------------------------------------------------------------- attention

def test_two_slot_logistic():
    """Two slots whose logits are 0 and 1 give the logistic weights
    1/(1+e), e/(1+e); a vote p on slot 2 scales its weight to pe/(1+pe)
    (KeepKV eq 6)."""
    d = 4
    q = np.array([[[1.0, 0, 0, 0]]])            # [U=1][G=1][d]
    k = np.array([[0.0, 0, 0, 0], [2.0, 0, 0, 0]])  # q.k/sqrt(4) = 0, 1
    v = np.array([[1.0, 2, 3, 4], [-1.0, 0.5, 0, 8]])
    for p in (1, 3):
        s = make_session(k, v, vote=[1, p])
        lse, f, probs = s.attend(q)
        w2 = p * math.e / (1 + p * math.e)
        assert lse[0, 0] == pytest.approx(math.log(1 + p * math.e), abs=1e-14)
        np.testing.assert_allclose(f[0, 0], (1 - w2) * v[0] + w2 * v[1], atol=1e-14)
        np.testing.assert_allclose(probs[0, :2], [1 - w2, w2], atol=1e-15)
        s.close()


def test_scale_is_inverse_sqrt_d():
    """d = 16: q = 4 e_0, k = e_0 gives logit 4/sqrt(16) = 1 against a zero key."""
    d = 16
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 4.0
    k = np.zeros((2, d)); k[1, 0] = 1.0
    v = np.zeros((2, d)); v[1, 0] = 1.0
    s = make_session(k, v)
    lse, f, _ = s.attend(q)
    assert f[0, 0, 0] == pytest.approx(math.e / (1 + math.e), abs=1e-15)
    s.close()


def test_uniform_logits_give_vote_weighted_mean():
    """q = 0: every logit is ln p_i, so weights are p_i / sum p and lse = ln sum p."""
    rng = np.random.default_rng(1)
    n, d, G = 9, 8, 3
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    p = rng.integers(1, 6, size=n)
    s = make_session(k, v, vote=p, G=G)
    lse, f, probs = s.attend(np.zeros((1, G, d)))
    for h in range(G):
        assert lse[0, h] == pytest.approx(math.log(p.sum()), abs=1e-14)
        np.testing.assert_allclose(f[0, h], (p[:, None] * v).sum(0) / p.sum(), atol=1e-14)
    np.testing.assert_allclose(probs[0, :n], p / p.sum(), atol=1e-15)
    s.close()


def test_vote_equals_duplication():
    """A slot with vote p gives the same output as p identical slots
    (KeepKV eq 6 and eq 23); its probability equals the duplicates' sum."""
    rng = np.random.default_rng(2)
    n, d, G = 7, 16, 4
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, G, d)))
    p = rng.integers(1, 5, size=n)
    a = make_session(k, v, vote=p, G=G)
    rep = np.repeat(np.arange(n), p)
    b = make_session(k[rep], v[rep], G=G)
    la, fa, pa = a.attend(q)
    lb, fb, pb = b.attend(q)
    np.testing.assert_allclose(la, lb, atol=1e-13)
    np.testing.assert_allclose(fa, fb, atol=1e-13)
    dup = np.zeros(n)
    np.add.at(dup, rep, pb[0, : rep.size])
    np.testing.assert_allclose(pa[0, :n], dup, atol=1e-14)
    a.close(); b.close()


def test_probs_match_softmax_and_sum_to_one():
    """Head-mean probabilities (InertiaKV eq 1) against scipy's softmax of
    q K^T / sqrt(d) + ln p, averaged over the group; they sum to 1."""
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    n, d, G = 33, 32, 4
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, G, d)))
    p = rng.integers(1, 9, size=n)
    s = make_session(k, v, vote=p, G=G)
    lse, f, probs = s.attend(q)
    A = softmax(q[0] @ k.T / math.sqrt(d) + np.log(p)[None, :], axis=1)
    np.testing.assert_allclose(probs[0, :n], A.mean(0), rtol=1e-12)
    np.testing.assert_allclose(f[0], A @ v, atol=1e-12)
    assert probs[0, :n].sum() == pytest.approx(1.0, abs=1e-13)
    s.close()


def test_split_decomposition():
    """Z = Z_R + Z_E and f = w_R f_R + w_E f_E with w_R = Z_R / Z
    (MomentKV sec 2, exact decomposition of the full output)."""
    rng = np.random.default_rng(4)
    n, d, G = 40, 16, 2
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, G, d)))
    p = rng.integers(1, 4, size=n)
    E = rng.permutation(n)[:13]
    R = np.setdiff1d(np.arange(n), E)
    full = make_session(k, v, vote=p, G=G)
    sR = make_session(k[R], v[R], vote=p[R], G=G)
    sE = make_session(k[E], v[E], vote=p[E], G=G)
    l, f, _ = full.attend(q)
    lR, fR, _ = sR.attend(q)
    lE, fE, _ = sE.attend(q)
    np.testing.assert_allclose(np.exp(l), np.exp(lR) + np.exp(lE), rtol=1e-13)
    wR = np.exp(lR - l)[..., None]
    np.testing.assert_allclose(f, wR * fR + (1 - wR) * fE, atol=1e-13)
    for s in (full, sR, sE):
        s.close()


def test_eviction_error_identity():
    """o' = (o - A_e v_e) / (1 - A_e) (KeepKV eq 3): evicting one slot and
    recomputing equals removing its share from the full output (G = 1, so the
    emitted probability is A_e)."""
    rng = np.random.default_rng(5)
    n, d = 21, 32
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, 1, d)))
    p = rng.integers(1, 4, size=n)
    for e in (0, 7, n - 1):
        full = make_session(k, v, vote=p)
        l, o, probs = full.attend(q)
        keep = np.setdiff1d(np.arange(n), [e])
        red = make_session(k[keep], v[keep], vote=p[keep])
        _, o2, _ = red.attend(q)
        Ae = probs[0, e]
        np.testing.assert_allclose(o2[0, 0], (o[0, 0] - Ae * v[e]) / (1 - Ae), atol=1e-13)
        full.close(); red.close()


# ---------------------------------------------------------------- utilities

def test_utility_rules_closed_forms():
    """InertiaKV eqs 2-4 with first observation m = s: constant s gives m = s
    under single and EMA; EMA after k refreshes of s' from m0 is
    alpha^k m0 + (1 - alpha^k) s'; cumulative is the running sum."""
    n, d = 5, 4
    k = np.zeros((n, d)); v = np.zeros((n, d))
    alpha = 0.9
    s0 = np.array([0.1, 0.2, 0.3, 0.25, 0.15])
    s1 = np.array([0.05, 0.4, 0.1, 0.3, 0.15])
    for rule in (O.RULE_SINGLE, O.RULE_CUMULATIVE, O.RULE_EMA):
        s = make_session(k, v, cap=n)
        probs = np.zeros((1, n))
        probs[0] = s0
        s.update_util(probs, rule, alpha)
        np.testing.assert_array_equal(s.slots()[3][0], s0)      # first observation
        for it in range(1, 6):
            probs[0] = s1
            s.update_util(probs, rule, alpha)
            m = s.slots()[3][0]
            if rule == O.RULE_SINGLE:
                np.testing.assert_array_equal(m, s1)
            elif rule == O.RULE_CUMULATIVE:
                np.testing.assert_allclose(m, s0 + it * s1, rtol=1e-15)
            else:
                np.testing.assert_allclose(m, alpha ** it * s0 + (1 - alpha ** it) * s1,
                                           rtol=1e-14)
        s.close()


def brute_force_victims(m, pos, scored, k):
    """Independent formulation: among all k-subsets of scored slots, those
    with the least total utility; among those, the one whose sorted positions
    are lexicographically smallest (evict the older token on equal utility)."""
    cand = [i for i in range(len(m)) if scored[i]]
    best = None
    for E in itertools.combinations(cand, k):
        key = (sum(m[i] for i in E), sorted(pos[i] for i in E))
        if best is None or key < best[0]:
            best = (key, E)
    return sorted(pos[i] for i in best[1])


@pytest.mark.parametrize("seed", range(12))
def test_selection_matches_brute_force(seed):
    """Lowest-utility eviction (InertiaKV sec 3.1; MomentKV Alg. 1 argmin
    loop) against subset enumeration, with ties from small integer utilities
    and some unscored (protected) slots."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(4, 12))
    L = int(rng.integers(1, n))
    d = 4
    s = O.DecodeSession(1, 1, d, n + 2)
    n_old = n - int(rng.integers(0, min(3, L) + 1))
    pos = rng.permutation(1000)[:n_old].astype(np.int32)
    s.load(0, np.zeros((n_old, d)), np.zeros((n_old, d)), pos=pos)
    util = rng.integers(0, 4, size=n_old) / 8.0      # exact ties
    probs = np.zeros((1, n + 2)); probs[0, :n_old] = util
    s.update_util(probs, O.RULE_SINGLE, 0.0)
    for j in range(n - n_old):                          # unscored newcomers
        s.append(np.zeros((1, d)), np.zeros((1, d)), 2000 + j)
    nn, P, _, M, SC = s.slots()
    k = n - L
    vic, nv, thr = s.select(L, k)
    assert nv[0] == k
    expect = brute_force_victims(M[0, :n], P[0, :n], SC[0, :n], k)
    assert sorted(vic[0, :k].tolist()) == expect
    s.close()


# ---------------------------------------------------------------- moments

def test_moments_match_two_pass_numpy():
    """Raw running sums (MomentKV App. A.1) reproduce the two-pass weighted
    mean and value-key covariance of the evicted set (numpy, centred first)."""
    rng = np.random.default_rng(6)
    n, d = 30, 8
    k = bf(rng.normal(1.0, 2.0, size=(n, d)))
    v = bf(rng.normal(-0.5, 1.0, size=(n, d)))
    p = rng.integers(1, 5, size=n)
    s = O.DecodeSession(1, 1, d, n)
    s.load(0, k, v, vote=p)
    E = rng.permutation(n)[:17]
    s.evict(E[None, :].astype(np.int32), np.array([E.size], np.int32))
    ne, mk, mv, C = s.moments()
    w = p[E].astype(float)
    muk = (w[:, None] * k[E]).sum(0) / w.sum()
    muv = (w[:, None] * v[E]).sum(0) / w.sum()
    Cn = ((w[:, None] * (v[E] - muv)).T @ (k[E] - muk)) / w.sum()
    assert ne[0] == w.sum()
    np.testing.assert_allclose(mk[0], muk, atol=1e-13)
    np.testing.assert_allclose(mv[0], muv, atol=1e-13)
    np.testing.assert_allclose(C[0], Cn, atol=1e-12)
    assert s.slots()[0][0] == n - E.size
    s.close()


def test_vote_fold_equals_duplicate_fold():
    rng = np.random.default_rng(7)
    n, d = 10, 8
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    p = rng.integers(1, 4, size=n)
    a = O.DecodeSession(1, 1, d, n)
    a.load(0, k, v, vote=p)
    rep = np.repeat(np.arange(n), p)
    b = O.DecodeSession(1, 1, d, rep.size)
    b.load(0, k[rep], v[rep])
    a.evict(np.arange(n, dtype=np.int32)[None], np.array([n], np.int32))
    b.evict(np.arange(rep.size, dtype=np.int32)[None], np.array([rep.size], np.int32))
    for x, y in zip(a.moments(), b.moments()):
        np.testing.assert_allclose(x, y, atol=1e-12)
    a.close(); b.close()


# ---------------------------------------------------------------- correction

def _corrected_vs_full(k, v, p, q, E, correction):
    n, d = k.shape
    G = q.shape[1]
    full = make_session(k, v, vote=p, G=G)
    _, f_full, _ = full.attend(q)
    full.close()
    s = make_session(k, v, vote=p, G=G)
    s.evict(np.asarray(E, np.int32)[None], np.array([len(E)], np.int32))
    o, fR, lz = s.output(q, correction)
    s.close()
    return o, fR, f_full


def test_correction_off_and_empty_moments_give_renormalized_output():
    """Correction off, or n_e = 0, returns f_R (MomentKV Algorithm 1: no
    evicted token yet means plain retained attention)."""
    rng = np.random.default_rng(8)
    n, d, G = 20, 16, 2
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, G, d)))
    p = np.ones(n, int)
    o, fR, _ = _corrected_vs_full(k, v, p, q, [3, 4, 5], O.CORR_OFF)
    np.testing.assert_array_equal(o, fR)
    o, fR, f_full = _corrected_vs_full(k, v, p, q, [], O.CORR_FIRST_ORDER)
    np.testing.assert_array_equal(o, fR)
    np.testing.assert_allclose(o, f_full, atol=1e-14)


@pytest.mark.parametrize("correction", [O.CORR_ZERO_ORDER, O.CORR_FIRST_ORDER])
def test_identical_evicted_keys_recover_full_output(correction):
    """If every evicted key is the same vector, all centred logits vanish:
    the Jensen bound is an equality (App. B.1) and fhat_E = v_bar = f_E, so
    the corrected output equals the full-cache output exactly."""
    rng = np.random.default_rng(9)
    n, d, G = 24, 16, 4
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    E = [2, 5, 11, 17, 20]
    k[E] = k[E[0]]
    p = rng.integers(1, 4, size=n)
    q = bf(rng.normal(size=(1, G, d)))
    o, fR, f_full = _corrected_vs_full(k, v, p, q, E, correction)
    np.testing.assert_allclose(o, f_full, atol=1e-13)
    assert np.abs(fR - f_full).max() > 1e-3       # plain renormalization is off


def test_zero_query_recovers_full_output():
    rng = np.random.default_rng(10)
    n, d, G = 24, 16, 2
    k, v = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    p = rng.integers(1, 4, size=n)
    o, fR, f_full = _corrected_vs_full(k, v, p, np.zeros((1, G, d)), [0, 1, 2, 9],
                                       O.CORR_FIRST_ORDER)
    np.testing.assert_allclose(o, f_full, atol=1e-14)


def _error_at_spread(sigma, correction, seed=11):
    rng = np.random.default_rng(seed)
    d, G, nR, nE = 16, 1, 12, 40
    A = rng.normal(size=(d, d)) / 4
    kR = rng.normal(size=(nR, d))
    xi = rng.normal(size=(nE, d))
    kE = sigma * xi
    k = np.vstack([kR, kE])
    v = np.vstack([rng.normal(size=(nR, d)), 0.5 + xi @ A.T + 0.02 * rng.normal(size=(nE, d))])
    k, v = bf(k), bf(v)
    q = bf(2.0 * rng.normal(size=(1, G, d)))
    E = list(range(nR, nR + nE))
    o, fR, f_full = _corrected_vs_full(k, v, np.ones(nR + nE, int), q, E, correction)
    return np.abs(o - f_full).max()


def test_first_order_error_is_second_order_in_spread():
    """The corrected output's error scales as sigma^2 (MomentKV sec 4.1 and
    App. A.2): halving the key spread quarters it.  The zero-order variant
    (v_bar only) is first order: halving sigma only halves it.  A sign error
    in the covariance term would also show up as first-order scaling."""
    e1 = [_error_at_spread(s, O.CORR_FIRST_ORDER) for s in (0.05, 0.025, 0.0125)]
    e0 = [_error_at_spread(s, O.CORR_ZERO_ORDER) for s in (0.05, 0.025, 0.0125)]
    for a, b in zip(e1, e1[1:]):
        assert 3.0 < a / b < 5.0, e1
    for a, b in zip(e0, e0[1:]):
        assert 1.6 < a / b < 2.6, e0
    assert e1[-1] < e0[-1] / 10


def test_jensen_lower_bound_tightness_and_self_regulation():
    """Zhat_E = n_e exp(q.k_bar/sqrt d) <= Z_E (MomentKV sec 4.2 eq 10,
    App. B.1).  Zhat_E is read back from the zero-order output
    o = w f_R + (1 - w) v_bar as Zhat_E = Z_R (1 - w) / w and compared with
    the exact Z_E of the evicted set:
      * w >= w_R and Zhat_E <= Z_E at every spread;
      * tightness: Z_E / Zhat_E - 1 ~ Var(delta) / 2 for a small spread, with
        delta_i = q.(k_i - k_bar)/sqrt(d) computed here in numpy (App. B.1);
      * self-regulation: Zhat_E / Z_E falls as the spread grows (App. B.2)."""
    rng = np.random.default_rng(12)
    d, nR, nE = 16, 10, 30
    kR = bf(rng.normal(size=(nR, d)))
    vR = bf(rng.normal(size=(nR, d)))
    vE = bf(rng.normal(size=(nE, d)) + 3.0)
    xi = rng.normal(size=(nE, d))
    q = bf(rng.normal(size=(1, 1, d)))
    ratios = []
    for sigma in (0.02, 0.04, 0.5, 2.0, 8.0):
        kE = bf(sigma * xi)
        k = np.vstack([kR, kE]); v = np.vstack([vR, vE])
        E = list(range(nR, nR + nE))
        s = make_session(k, v)
        s.evict(np.asarray(E, np.int32)[None], np.array([nE], np.int32))
        o, fR, lzR = s.output(q, O.CORR_ZERO_ORDER)
        s.close()
        vbar = vE.mean(0)
        dvec = fR[0, 0] - vbar
        w = float((o[0, 0] - vbar) @ dvec / (dvec @ dvec))
        sE = make_session(kE, vE)
        lE, _, _ = sE.attend(q)
        sE.close()
        wR = 1.0 / (1.0 + math.exp(lE[0, 0] - lzR[0, 0]))
        assert w >= wR - 1e-12
        log_zhat = lzR[0, 0] + math.log((1 - w) / w)
        assert log_zhat <= lE[0, 0] + 1e-12
        ratios.append(math.exp(log_zhat - lE[0, 0]))
        if sigma <= 0.04:
            delta = (kE - kE.mean(0)) @ q[0, 0] / math.sqrt(d)
            half_var = 0.5 * np.mean(delta ** 2)
            assert (1.0 / ratios[-1] - 1.0) == pytest.approx(half_var, rel=0.05)
    assert all(a > b for a, b in zip(ratios, ratios[1:])), ratios
    assert ratios[-1] < 1e-3


# ---------------------------------------------------------------- pipeline

def test_no_eviction_when_budget_covers_everything():
    """With L >= N + steps nothing is evicted: the output is plain attention
    over every token and the moments stay zero."""
    rng = np.random.default_rng(13)
    U, N, d, G, S = 2, 12, 8, 2, 4
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    res = O.decode_generation(kp, vp, qs, ks, vs, L=N + S, rule=O.RULE_EMA,
                              alpha=0.9, T=1, correction=O.CORR_FIRST_ORDER)
    for r in res:
        assert (r["applied_nvict"] == 0).all()
        np.testing.assert_allclose(r["o"], r["f_all"], atol=1e-14)
        assert (r["moments"][0] == 0).all()


def test_generation_invariants_and_lazy_refresh():
    """Whole decode loop: after every step each unit holds min(L, ...) slots;
    step 1 evicts N + 1 - L, later steps one each; under a refresh period T
    the utilities only change on refresh steps (InertiaKV-Lazy), so with T
    longer than the run every surviving prefill slot keeps its step-1 score
    (Score-Free)."""
    rng = np.random.default_rng(14)
    U, N, d, G, S, L = 2, 20, 8, 2, 6, 8
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    sess = O.DecodeSession(U, G, d, N + S)
    for u in range(U):
        sess.load(u, kp[u], vp[u])
    step1 = None
    for s in range(S):
        t = s + 1
        r = O.decode_step(sess, t, N + t - 1, qs[s], ks[s], vs[s], L=L,
                          rule=O.RULE_EMA, alpha=0.9, T=S + 5,
                          correction=O.CORR_FIRST_ORDER)
        n, pos, _, util, scored = sess.slots()
        assert (n == L).all()
        assert (r["applied_nvict"] == (N + 1 - L if t == 1 else 1)).all()
        assert r["refresh"] == (t == 1)
        if t == 1:
            # before the step-1 eviction slot i held position i
            step1 = {(u, i): r["probs"][u, i] for u in range(U) for i in range(N + 1)}
        for u in range(U):
            for i in range(L):
                if scored[u, i]:
                    assert util[u, i] == step1[(u, int(pos[u, i]))]
                else:
                    assert pos[u, i] >= N + 1     # appended after the refresh
    sess.close()


def test_score_free_evicts_in_step1_order():
    """Score-Free (InertiaKV abstract, sec 1: score the full context once at
    the first decode step, then keep that ranking): with T = 0 the victims
    of the whole run are the step-1 head-mean softmax ranking, lowest first
    (ties to the older token), N + 1 - L at step 1 and then one per step,
    and no token appended after step 1 is ever evicted.  The ranking is
    brute-forced here with numpy's softmax over the step-1 cache."""
    rng = np.random.default_rng(15)
    U, N, d, G, S, L = 2, 24, 8, 4, 9, 12
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    res = O.decode_generation(kp, vp, qs, ks, vs, L=L, rule=O.RULE_EMA,
                              alpha=0.9, T=0, correction=O.CORR_FIRST_ORDER)
    assert [r["refresh"] for r in res] == [True] + [False] * (S - 1)
    for u in range(U):
        keys = np.concatenate([kp[u], ks[0, u][None]])          # positions 0..N
        x = qs[0, u] @ keys.T / math.sqrt(d)                    # [G][N+1]
        a = np.exp(x - x.max(axis=1, keepdims=True))
        s1 = (a / a.sum(axis=1, keepdims=True)).mean(axis=0)
        order = sorted(range(N + 1), key=lambda i: (s1[i], i))
        got = []
        for t, r in enumerate(res, start=1):
            nv = int(r["applied_nvict"][u])
            assert nv == (N + 1 - L if t == 1 else 1)
            got.append(sorted(int(p) for p in r["applied_victims"][u, :nv]))
        assert got[0] == sorted(order[:N + 1 - L])
        assert [g[0] for g in got[1:]] == order[N + 1 - L:N + 1 - L + S - 1]


# ---------------------------------------------------------------- moment-informed eviction

def _two_token_moments_session(G=1):
    """One unit whose eviction set is {(k1, v1), (k2, v2)} (integer vectors),
    so that k_bar = (k1 + k2)/2, dk = (k1 - k2)/2, C = dv dk^T (population
    covariance of two points), plus retained slots appended afterwards."""
    d = 16
    k1 = np.zeros(d); k1[:4] = [3, 1, 1, 1]          # dk = (1,1,1,1,0..), |dk|^2 = 4 = sqrt(d)
    k2 = np.zeros(d); k2[:4] = [1, -1, -1, -1]
    v1 = np.zeros(d); v1[4:6] = [2, 0]
    v2 = np.zeros(d); v2[4:6] = [0, 2]                # dv = (1, -1) in dims 4, 5
    s = O.DecodeSession(1, G, d, 8)
    s.load(0, np.stack([k1, k2]), np.stack([v1, v2]))
    s.evict(np.array([[0, 1]], np.int32), np.array([2], np.int32))
    return s, d, (k1 + k2) / 2, (k1 - k2) / 2, (v1 + v2) / 2, (v1 - v2) / 2


def test_mi_residual_closed_form_and_exact_prediction():
    """MomentKV moment residual r = v - v_bar - C (k - k_bar) / sqrt(d) with
    the two-token eviction set: C (k - k_bar)/sqrt(d) = dv (dk . (k - k_bar))
    / sqrt(d).  A token at k_bar + 2 dk with value v_bar + 2 dv is predicted
    exactly (score 0); another one's residual norm is the closed form."""
    s, d, kb, dk, vb, dv = _two_token_moments_session()
    ka, va = kb + 2 * dk, vb + 2 * dv                 # on the affine model
    kx, vx = kb + dk, vb + 3 * dv                     # off it by dv
    ky = kb.copy(); ky[8] = 5.0
    vy = vb.copy(); vy[9] = 2.0                       # dk . (ky - kb) = 0
    for j, (kk, vv) in enumerate([(ka, va), (kx, vx), (ky, vy)]):
        s.append(kk[None], vv[None], 10 + j)
    probs = np.zeros((1, 8)); probs[0, :3] = [0.5, 0.25, 0.125]
    sc = s.mi_scores(probs)[0, :3]
    assert sc[0] == 0.0
    assert sc[1] == pytest.approx(0.25 * 2.0 * np.linalg.norm(dv), rel=1e-14)
    assert sc[2] == pytest.approx(0.125 * np.linalg.norm(vy - vb), rel=1e-14)
    s.close()


def test_mi_scores_without_moments_are_weight_times_value_norm():
    """n_e = 0: v_bar and S_tilde are zero, r = v and the score is
    alpha ||v|| (MomentKV Algorithm 1, phase 1)."""
    rng = np.random.default_rng(21)
    k, v = bf(rng.normal(size=(9, 8))), bf(rng.normal(size=(9, 8)))
    s = make_session(k, v)
    probs = np.zeros((1, s.cap)); probs[0, :9] = rng.random(9)
    sc = s.mi_scores(probs)[0, :9]
    np.testing.assert_allclose(sc, probs[0, :9] * np.linalg.norm(v, axis=1), rtol=1e-14)
    s.close()


def test_mi_residual_matches_numpy_covariance_and_is_shift_invariant():
    """Residual norms against numpy's two-pass population covariance of the
    evicted set (np.cov, bias=True), and invariant when every key, or every
    value, is shifted by one common vector (the centring)."""
    rng = np.random.default_rng(22)
    d, nE, nR = 8, 6, 5
    # quarter-integers: the shifted arrays stay exact in bf16
    base_k = rng.integers(-8, 9, size=(nE + nR, d)) / 4.0
    base_v = rng.integers(-8, 9, size=(nE + nR, d)) / 4.0
    shift = rng.integers(-3, 4, size=d).astype(float)

    def scores(k, v):
        s = make_session(k, v, cap=nE + nR + 2)
        s.evict(np.arange(nE, dtype=np.int32)[None], np.array([nE], np.int32))
        probs = np.ones((1, s.cap))
        out = s.mi_scores(probs)[0, :nR]
        s.close()
        return out
    ref = scores(base_k, base_v)
    KE, VE = base_k[:nE], base_v[:nE]
    C = np.cov(np.hstack([VE, KE]).T, bias=True)[:d, d:]
    R = base_v[nE:] - VE.mean(0) - (base_k[nE:] - KE.mean(0)) @ C.T / math.sqrt(d)
    np.testing.assert_allclose(ref, np.linalg.norm(R, axis=1), rtol=1e-12)
    np.testing.assert_allclose(scores(base_k + shift, base_v), ref, rtol=1e-12)
    np.testing.assert_allclose(scores(base_k, base_v + shift), ref, rtol=1e-12)


def _numpy_mi_round(k, v, p, q, evk, evv, evp):
    """Scores of one round of MomentKV Algorithm 1 phase 1, restated with
    numpy / scipy: alpha = head mean of the vote-weighted softmax over the
    slots present, moments of the evicted tokens by numpy's weighted
    two-pass covariance (fweights = votes), residual and score."""
    from scipy.special import softmax
    d = k.shape[1]
    x = q @ k.T / math.sqrt(d) + np.log(p)[None, :]          # [G][n]
    alpha = softmax(x, axis=1).mean(axis=0)
    if len(evp) == 0:
        r = v
    else:
        w = np.asarray(evp)
        mk = np.average(evk, axis=0, weights=w)
        mv = np.average(evv, axis=0, weights=w)
        C = np.cov(np.hstack([evv, evk]).T, fweights=w, bias=True)[:d, d:]
        r = v - mv - (k - mk) @ C.T / math.sqrt(d)
    return alpha * np.linalg.norm(r, axis=1)


def test_mi_greedy_rounds_are_the_argmin_of_independent_scores():
    """MomentKV Algorithm 1 phase 1 with k > 1: every round removes the
    slot whose score, recomputed from scratch (numpy: softmax over the
    slots still present, weighted covariance of every token evicted so far)
    is lowest among all slots present, by brute force over the candidates,
    ties to the smaller position; votes weight the fold (KeepKV eq 6)."""
    rng = np.random.default_rng(31)
    for trial in range(12):
        d, G = 8, 2
        n = int(rng.integers(6, 13))
        k_ = int(rng.integers(2, 5))
        L = n - k_
        kk = bf(rng.normal(size=(n, d)))
        vv = bf(rng.normal(size=(n, d)))
        p = rng.integers(1, 4, size=n).astype(np.int32)
        q = bf(rng.normal(size=(1, G, d)))
        s = O.DecodeSession(1, G, d, n + 2)
        s.load(0, kk, vv, p)
        g = s.mi_greedy(q, L, k_)
        assert g["nvict"][0] == k_
        present = list(range(n))
        evk, evv, evp = [], [], []
        for r in range(k_):
            sc = _numpy_mi_round(kk[present], vv[present], p[present].astype(float), q[0],
                                 np.array(evk).reshape(-1, d), np.array(evv).reshape(-1, d), evp)
            j = min(range(len(present)), key=lambda i: (sc[i], present[i]))
            assert g["victims"][0, r] == present[j], (trial, r)
            assert g["best"][0, r] == pytest.approx(sc[j], rel=1e-9, abs=1e-300)
            evk.append(kk[present[j]]); evv.append(vv[present[j]]); evp.append(float(p[present[j]]))
            del present[j]
        s.close()


def test_mi_greedy_refolds_between_rounds():
    """A case where scoring once and taking the two lowest differs from the
    page's loop.  Logits 0, 1, 1/2, 2, 2 (q = 2 e_0, d = 4) and unit values
    v_A = v_B = e_0, v_C = e_1, v_D = e_2, v_E = e_3, nothing evicted yet:
    the first scores are alpha ||v|| with the order A < C < B < D = E.
    Round 1 evicts A; folding it makes (v_bar, S_tilde) = (e_0, 0), so B's
    residual is exactly 0 and round 2 evicts B, not C."""
    d = 4
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 2.0
    k = np.zeros((5, d)); k[:, 0] = [0.0, 1.0, 0.5, 2.0, 2.0]
    v = np.zeros((5, d)); v[0, 0] = v[1, 0] = 1.0; v[2, 1] = 1.0; v[3, 2] = 1.0; v[4, 3] = 1.0
    s = make_session(k, v)
    g = s.mi_greedy(q, 3, 2)
    assert g["victims"][0, :2].tolist() == [0, 1]
    assert g["best"][0, 1] == 0.0
    e = np.exp([0.0, 1.0, 0.5, 2.0, 2.0])
    np.testing.assert_allclose(g["scores0"][0, :5], e / e.sum(), rtol=1e-14)
    s.close()


def test_mi_greedy_equals_one_round_at_a_time():
    """k rounds in one call are k calls of one round each with the budget
    lowered by one (the same query, no token appended in between)."""
    rng = np.random.default_rng(33)
    d, G, n, k_ = 8, 4, 11, 4
    kk, vv = bf(rng.normal(size=(n, d))), bf(rng.normal(size=(n, d)))
    q = bf(rng.normal(size=(1, G, d)))
    a = make_session(kk, vv, G=G)
    b = make_session(kk, vv, G=G)
    ga = a.mi_greedy(q, n - k_, k_)
    order = [int(b.mi_greedy(q, n - 1 - r, 1)["victims"][0, 0]) for r in range(k_)]
    assert ga["victims"][0, :k_].tolist() == order
    for x, y in zip(a.moments(), b.moments()):
        np.testing.assert_array_equal(x, y)
    a.close(); b.close()


def test_mi_generation_evicts_the_lowest_score():
    """Decode loop with the moment-informed rule: every step re-scores (the
    new token included) and evicts the slot with the lowest alpha ||r||
    (ties to the older position), checked by brute force on the step's
    scores; the first step removes several slots, one argmin and one fold
    at a time (MomentKV Algorithm 1 phase 1)."""
    rng = np.random.default_rng(23)
    U, N, d, G, S, L = 2, 16, 8, 2, 6, 10
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    sess = O.DecodeSession(U, G, d, N + S)
    for u in range(U):
        sess.load(u, kp[u], vp[u])
    for s_ in range(S):
        t = s_ + 1
        n0, pos0, _, _, _ = sess.slots()
        r = O.decode_step(sess, t, N + t - 1, qs[s_], ks[s_], vs[s_], L=L, rule=O.RULE_MI,
                          alpha=0.9, T=1, correction=O.CORR_FIRST_ORDER)
        assert r["refresh"]
        for u in range(U):
            n = int(n0[u]) + 1
            k = n - L
            assert r["applied_nvict"][u] == k
            if k == 1:
                pos = np.append(pos0[u, : n0[u]], N + t - 1)
                sc = r["mi_scores"][u, :n]
                want = min(range(n), key=lambda i: (sc[i], pos[i]))
                assert r["applied_victims"][u, 0] == pos[want]
            assert r["mi_used"][u, :k].tolist() == r["mi_best"][u, :k].tolist()
    sess.close()


def test_per_unit_budgets_select_like_single_units():
    """Budgets per unit (a cache handed over from a prefill scorer keeps each
    unit at its own length) select, per unit, what a one-unit session with
    that budget selects."""
    rng = np.random.default_rng(51)
    U, n, d = 3, 12, 4
    Lu = np.array([9, 11, 5], np.int32)
    k, v = bf(rng.normal(size=(U, n, d))), bf(rng.normal(size=(U, n, d)))
    util = rng.random((U, n))
    s = O.DecodeSession(U, 1, d, n + 2)
    for u in range(U):
        s.load(u, k[u], v[u])
        s.set_util(u, util[u])
    vic, nv, _ = s.select(Lu, 8)
    for u in range(U):
        one = make_session(k[u], v[u])
        one.set_util(0, util[u])
        v1, n1, _ = one.select(int(Lu[u]), 8)
        assert nv[u] == n1[0] == n - Lu[u]
        assert vic[u, : nv[u]].tolist() == v1[0, : n1[0]].tolist()
        one.close()
    s.close()


# ------------------------------------------------------ layer-chained EMA

def _chained_session(rng, B, NL, Hkv, n, d=4):
    U = B * NL * Hkv
    k = bf(rng.normal(size=(B, n, d)))
    s = O.DecodeSession(U, 1, d, n + 2)
    for u in range(U):
        b = u // (NL * Hkv)
        s.load(u, k[b], k[b])            # every unit of a sequence: the same positions
    return s, U


def test_chained_ema_closed_form_over_layers():
    """One refresh from utilities m0 with layer means s_l: the state passes
    the layers in order, m = alpha^NL m0 + sum_l (1 - alpha) alpha^(NL-1-l) s_l,
    s_l the mean over the layer's KV units of their head-mean probabilities
    (InertiaKV sec 3.1: all H heads of the layer); every unit of the
    sequence gets the same utility."""
    rng = np.random.default_rng(61)
    B, NL, Hkv, n, al = 2, 3, 2, 5, 0.7
    s, U = _chained_session(rng, B, NL, Hkv, n)
    m0 = rng.random((B, n))
    for u in range(U):
        s.set_util(u, m0[u // (NL * Hkv)])
    probs = np.zeros((U, s.cap))
    probs[:, :n] = rng.random((U, n))
    s.update_util_chained(probs, NL, Hkv, al)
    util = s.slots()[3]
    for b in range(B):
        sl = [probs[b * NL * Hkv + l * Hkv: b * NL * Hkv + (l + 1) * Hkv, :n].mean(axis=0)
              for l in range(NL)]
        want = al ** NL * m0[b] + sum((1 - al) * al ** (NL - 1 - l) * sl[l] for l in range(NL))
        for q in range(NL * Hkv):
            np.testing.assert_allclose(util[b * NL * Hkv + q, :n], want, rtol=1e-14)
    s.close()


def test_chained_ema_first_observation_and_one_layer():
    """An unscored slot starts from the first layer's mean (the plain EMA's
    first observation), then chains; with one layer and one KV head the
    chained rule is the per-unit EMA."""
    rng = np.random.default_rng(62)
    NL, Hkv, n, al = 4, 1, 6, 0.9
    s, U = _chained_session(rng, 1, NL, Hkv, n)
    probs = np.zeros((U, s.cap)); probs[:, :n] = rng.random((U, n))
    s.update_util_chained(probs, NL, Hkv, al)
    m = probs[0, :n].copy()
    for l in range(1, NL):
        m = al * m + (1 - al) * probs[l, :n]
    np.testing.assert_allclose(s.slots()[3][0, :n], m, rtol=1e-14)
    s.close()
    a, U = _chained_session(rng, 1, 1, 1, n)
    b, _ = _chained_session(rng, 1, 1, 1, n)
    for t in range(3):
        p = np.zeros((1, a.cap)); p[0, :n] = rng.random(n)
        a.update_util_chained(p, 1, 1, al)
        b.update_util(p, O.RULE_EMA, al)
    np.testing.assert_array_equal(a.slots()[3], b.slots()[3])
    a.close(); b.close()


def test_chained_generation_evicts_the_same_positions_everywhere():
    """A whole decode run under the chained rule: every unit of a sequence
    evicts the same positions each step, the lowest chained utility (brute
    force over the sequence's slots)."""
    rng = np.random.default_rng(63)
    B, NL, Hkv, G, N, d, S, L = 2, 3, 2, 2, 12, 8, 6, 8
    U = B * NL * Hkv
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    sess = O.DecodeSession(U, G, d, N + S)
    for u in range(U):
        sess.load(u, kp[u], vp[u])
    for s_ in range(S):
        t = s_ + 1
        r = O.decode_step(sess, t, N + t - 1, qs[s_], ks[s_], vs[s_], L=L, rule=O.RULE_CHAINED,
                          alpha=0.8, T=1, correction=O.CORR_FIRST_ORDER, chain=(NL, Hkv))
        for b in range(B):
            sets = {tuple(sorted(r["applied_victims"][u, : r["applied_nvict"][u]].tolist()))
                    for u in range(b * NL * Hkv, (b + 1) * NL * Hkv)}
            assert len(sets) == 1
    sess.close()
