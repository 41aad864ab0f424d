"""Pins of the fp64 oracle's LaProx prefill scorer ("Reformulating KV Cache
Eviction Problem for Long-Context LLM Inference", arXiv 2605.07234, key
designs 1-3) against closed forms, numpy and brute force."""
import itertools
import math

import numpy as np
import pytest

from oracle import oracle as O


def bf(x):
    return O.bf16_round(x)


def test_gram_route_matches_direct_projection():
    """r_i = sqrt(v^T W_g W_g^T v) equals ||v W_g|| computed by numpy's matmul
    and by the oracle's direct route, W_g the sum of the group's W_O slices."""
    rng = np.random.default_rng(0)
    NL, Hq, Hkv, d, N = 2, 4, 2, 8, 20
    D = Hq * d
    W = bf(rng.normal(0, 0.2, size=(NL, Hq * d, D)))
    V = bf(rng.normal(size=(NL, Hkv, N, d)))
    Gram = O.prefill_gram(W, NL, Hq, Hkv, d)
    r = O.prefill_rownorm(V, Gram, NL, Hkv, d, N)
    G = Hq // Hkv
    for l in range(NL):
        for g in range(Hkv):
            Wg = sum(W[l, h * d:(h + 1) * d, :] for h in range(g * G, (g + 1) * G))
            np.testing.assert_allclose(r[l, g], np.linalg.norm(V[l, g] @ Wg, axis=1), rtol=1e-12)
            tok = np.array([0, 7, N - 1], np.int32)
            direct = O.prefill_rownorm_direct(V, W, Hq, Hkv, d, N, l, g, tok)
            np.testing.assert_allclose(direct, r[l, g, tok], rtol=1e-12)


def test_orthonormal_projection_scales_norm():
    """If W_g = c [I | 0] (orthonormal rows times c) then r_i = c ||v_i||."""
    rng = np.random.default_rng(1)
    NL, Hq, Hkv, d, N = 1, 4, 1, 8, 6
    D = Hq * d
    W = np.zeros((NL, Hq * d, D))
    for h in range(Hq):
        W[0, h * d:(h + 1) * d, :d] = 0.5 * np.eye(d)      # sum over 4 heads: 2 I
    V = bf(rng.normal(size=(NL, Hkv, N, d)))
    r = O.prefill_rownorm(V, O.prefill_gram(W, NL, Hq, Hkv, d), NL, Hkv, d, N)
    np.testing.assert_allclose(r[0, 0], 2.0 * np.linalg.norm(V[0, 0], axis=1), rtol=1e-14)


def test_uniform_window_attention_closed_form():
    """q = 0: window row j (position N-w+j) spreads weight 1/(N-w+j+1) over
    the keys it sees, so c_i = sqrt(sum over rows that see key i of
    1/(N-w+j+1)^2); this pins the causal mask and the group mean."""
    NL, Hq, Hkv, d, N, w = 1, 4, 2, 8, 12, 5
    rng = np.random.default_rng(2)
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    q = np.zeros((NL, Hq, w, d))
    c = O.prefill_colnorm(q, K, NL, Hq, Hkv, d, N, w)
    for i in range(N):
        expect = math.sqrt(sum(1.0 / (N - w + j + 1) ** 2 for j in range(w) if i <= N - w + j))
        np.testing.assert_allclose(c[0, :, i], expect, rtol=1e-13)


def test_dominant_key_gives_sqrt_window():
    """Every window row of every head putting all its weight on key i* gives
    A_bar[:, i*] = 1, so c_{i*} = sqrt(w) and the other columns vanish."""
    NL, Hq, Hkv, d, N, w = 1, 4, 1, 16, 40, 8
    K = np.zeros((NL, Hkv, N, d))
    istar = 13
    K[0, 0, istar, 0] = 64.0
    q = np.zeros((NL, Hq, w, d)); q[..., 0] = 8.0            # logit 128 vs 0
    c = O.prefill_colnorm(q, K, NL, Hq, Hkv, d, N, w)
    assert c[0, 0, istar] == pytest.approx(math.sqrt(w), rel=1e-12)
    assert np.delete(c[0, 0], istar).max() < 1e-40


def test_colnorm_matches_scipy_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    NL, Hq, Hkv, d, N, w = 1, 6, 2, 8, 15, 4
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    q = bf(rng.normal(size=(NL, Hq, w, d)))
    c = O.prefill_colnorm(q, K, NL, Hq, Hkv, d, N, w)
    G = Hq // Hkv
    for g in range(Hkv):
        Abar = np.zeros((w, N))
        for h in range(g * G, (g + 1) * G):
            x = q[0, h] @ K[0, g].T / math.sqrt(d)
            mask = np.arange(N)[None, :] > (N - w + np.arange(w))[:, None]
            x[mask] = -np.inf
            Abar += softmax(x, axis=1) / G
        np.testing.assert_allclose(c[0, g], np.linalg.norm(Abar, axis=0), rtol=1e-12)


def test_layer_normalization_sums_to_one():
    rng = np.random.default_rng(4)
    NL, Hkv, N = 3, 2, 10
    c = rng.random((NL, Hkv, N)); r = rng.random((NL, Hkv, N)) * 10 ** np.arange(NL)[:, None, None]
    res = O.prefill_select(c, r, 7, normalize=True)
    np.testing.assert_allclose(res["s"].sum(axis=(1, 2)), 1.0, rtol=1e-14)
    raw = O.prefill_select(c, r, 7, normalize=False)
    np.testing.assert_allclose(raw["s"], c * r, rtol=0)


@pytest.mark.parametrize("seed", range(10))
def test_global_topk_matches_brute_force(seed):
    """Model-wide top-K (LaProx key design 3) against subset enumeration:
    the K-subset of largest total score, ties broken towards the
    lexicographically smallest flat indices."""
    rng = np.random.default_rng(50 + seed)
    NL, Hkv, N = 2, 2, int(rng.integers(2, 4))
    M = NL * Hkv * N
    Kb = int(rng.integers(1, M))
    c = rng.integers(1, 4, size=(NL, Hkv, N)).astype(float)
    r = np.ones((NL, Hkv, N))
    res = O.prefill_select(c, r, Kb, normalize=True)
    from fractions import Fraction
    p = (c * r).astype(int)
    s = [Fraction(int(p.ravel()[j]), int(p[j // (Hkv * N)].sum())) for j in range(M)]
    best = None
    for S in itertools.combinations(range(M), Kb):
        key = (-sum(s[j] for j in S), list(S))     # exact rational sums
        if best is None or key < best[0]:
            best = (key, S)
    assert sorted(res["idx"].tolist()) == list(best[1])
    assert res["keep"].ravel().nonzero()[0].tolist() == list(best[1])
    assert res["counts"].sum() == Kb
    np.testing.assert_array_equal(res["counts"], res["keep"].sum(axis=2))


def _brute_segment_topk(s, lo, hi, k):
    """The k-subset of [lo, hi) with the largest total score, ties towards
    the lexicographically smallest indices (exact rationals)."""
    best = None
    for S in itertools.combinations(range(lo, hi), k):
        key = (-sum(s[j] for j in S), list(S))
        if best is None or key < best[0]:
            best = (key, S)
    return list(best[1])


@pytest.mark.parametrize("alloc", [O.ALLOC_LAYER, O.ALLOC_HEAD])
@pytest.mark.parametrize("seed", range(6))
def test_segment_allocations_match_brute_force(alloc, seed):
    """LaProx allocation ablation: head-flatten only (a B_total / NL budget
    per layer over its heads and tokens) and uniform per head (B_total /
    (NL Hkv) per KV head) against subset enumeration within each segment,
    with exact rational scores and ties."""
    from fractions import Fraction
    rng = np.random.default_rng(80 + seed)
    NL, Hkv, N = 2, 2, 3
    M = NL * Hkv * N
    nseg = NL if alloc == O.ALLOC_LAYER else NL * Hkv
    kseg = int(rng.integers(1, M // nseg))
    c = rng.integers(1, 4, size=(NL, Hkv, N)).astype(float)
    r = np.ones((NL, Hkv, N))
    res = O.prefill_select(c, r, kseg * nseg, normalize=True, alloc=alloc)
    p = (c * r).astype(int)
    s = [Fraction(int(p.ravel()[j]), int(p[j // (Hkv * N)].sum())) for j in range(M)]
    seg = M // nseg
    want = []
    for q in range(nseg):
        want += _brute_segment_topk(s, q * seg, (q + 1) * seg, kseg)
    assert res["keep"].ravel().nonzero()[0].tolist() == want
    assert res["idx"].tolist() == want
    np.testing.assert_array_equal(res["counts"], res["keep"].sum(axis=2))
    if alloc == O.ALLOC_HEAD:
        assert (res["counts"] == kseg).all()
    else:
        assert (res["counts"].sum(axis=1) == kseg).all()


def test_allocations_agree_on_one_segment():
    """With one layer and one KV head every allocation is the same top-K;
    with one layer the global and per-layer selections coincide."""
    rng = np.random.default_rng(9)
    c1, r1 = rng.random((1, 1, 40)), rng.random((1, 1, 40))
    sets = [O.prefill_select(c1, r1, 11, alloc=a)["idx"].tolist()
            for a in (O.ALLOC_GLOBAL, O.ALLOC_LAYER, O.ALLOC_HEAD)]
    assert sets[0] == sets[1] == sets[2]
    c2, r2 = rng.random((1, 4, 30)), rng.random((1, 4, 30))
    assert (O.prefill_select(c2, r2, 20, alloc=O.ALLOC_GLOBAL)["idx"].tolist()
            == O.prefill_select(c2, r2, 20, alloc=O.ALLOC_LAYER)["idx"].tolist())


def test_segment_budget_must_divide():
    c, r = np.ones((2, 2, 5)), np.ones((2, 2, 5))
    with pytest.raises(ValueError):
        O.prefill_select(c, r, 7, alloc=O.ALLOC_HEAD)


# ---------------------------------------------------------------- KeepKV windowed EMA init

def _window_case(seed, NL=1, Hq=4, Hkv=2, N=20, w=5, d=8, zero_q=False):
    rng = np.random.default_rng(seed)
    q = np.zeros((NL, Hq, w, d)) if zero_q else O.bf16_round(rng.normal(size=(NL, Hq, w, d)))
    K = O.bf16_round(rng.normal(size=(NL, Hkv, N, d)))
    return q, K


@pytest.mark.parametrize("alpha", [0.0, 0.5, 0.9])
def test_ema_init_mass_is_one_minus_alpha_to_the_w(alpha):
    """Every window row is a probability distribution, so the initialized
    utilities of a (layer, KV head) sum to sum_j (1 - a) a^(w-1-j) =
    1 - a^w (the bias KeepKV's eq 14 corrects)."""
    q, K = _window_case(31)
    S = O.prefill_ema_init(q, K, 1, 4, 2, 8, 20, 5, alpha)
    np.testing.assert_allclose(S.sum(axis=2), 1.0 - alpha ** 5, rtol=1e-13)


def test_ema_init_alpha_zero_is_the_last_query():
    """alpha = 0 keeps only the last window query's group-mean attention
    (scipy softmax, causal: it sees every key)."""
    from scipy.special import softmax
    q, K = _window_case(32)
    S = O.prefill_ema_init(q, K, 1, 4, 2, 8, 20, 5, 0.0)
    for g in range(2):
        x = np.stack([K[0, g] @ q[0, h, -1] / math.sqrt(8) for h in (2 * g, 2 * g + 1)])
        np.testing.assert_allclose(S[0, g], softmax(x, axis=1).mean(axis=0), rtol=1e-12)


def test_ema_init_zero_query_closed_form():
    """q = 0: window query j attends uniformly to its N - w + j + 1 visible
    keys, so S_i = sum over the queries that see i of (1 - a) a^(w-1-j) /
    (N - w + j + 1)."""
    N, w, a = 20, 5, 0.7
    q, K = _window_case(33, zero_q=True)
    S = O.prefill_ema_init(q, K, 1, 4, 2, 8, N, w, a)
    want = np.array([sum((1 - a) * a ** (w - 1 - j) / (N - w + j + 1)
                         for j in range(w) if i <= N - w + j) for i in range(N)])
    np.testing.assert_allclose(S[0, 0], want, rtol=1e-13)
    np.testing.assert_allclose(S[0, 1], want, rtol=1e-13)


def test_initialized_utilities_continue_the_ema_at_step_one():
    """A slot carrying an initialized utility is scored: the first decode
    step applies m = a m0 + (1 - a) s instead of m = s."""
    rng = np.random.default_rng(34)
    k, v = O.bf16_round(rng.normal(size=(6, 8))), O.bf16_round(rng.normal(size=(6, 8)))
    s = O.DecodeSession(1, 1, 8, 8)
    s.load(0, k, v)
    m0 = rng.random(6)
    s.set_util(0, m0)
    probs = np.zeros((1, 8)); probs[0, :6] = rng.random(6)
    s.update_util(probs, O.RULE_EMA, 0.9)
    _, _, _, util, scored = s.slots()
    np.testing.assert_allclose(util[0, :6], 0.9 * m0 + 0.1 * probs[0, :6], rtol=1e-15)
    assert scored[0, :6].all()
    s.close()


# ------------------------------------------------------- SnapKV protocol

def test_window_colsum_unit_weights_sum_to_the_window():
    """With every row weight 1 (SnapKV's accumulated window attention) each
    window row's group-mean softmax sums to 1 over the keys it sees, so the
    accumulated scores of a (layer, KV head) sum to w."""
    rng = np.random.default_rng(41)
    NL, Hq, Hkv, d, N, w = 2, 8, 2, 16, 40, 6
    q = bf(rng.normal(size=(NL, Hq, w, d)))
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    S = O.prefill_window_colsum(q, K, NL, Hq, Hkv, d, N, w, np.ones(w))
    np.testing.assert_allclose(S.sum(axis=2), w, rtol=1e-13)


def test_window_colsum_single_row_is_scipy_group_softmax():
    """A weight vector selecting window row j alone gives the group mean of
    the G heads' causal softmax of that row (scipy), keys past its position
    zero; a weighted sum is linear in the weights."""
    from scipy.special import softmax
    rng = np.random.default_rng(42)
    NL, Hq, Hkv, d, N, w = 1, 4, 1, 8, 24, 5
    q = bf(rng.normal(size=(NL, Hq, w, d)))
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    j = 2
    e = np.zeros(w); e[j] = 1.0
    S = O.prefill_window_colsum(q, K, NL, Hq, Hkv, d, N, w, e)
    last = N - w + j
    ref = np.mean([softmax(q[0, h, j] @ K[0, 0, : last + 1].T / math.sqrt(d)) for h in range(Hq)],
                  axis=0)
    np.testing.assert_allclose(S[0, 0, : last + 1], ref, rtol=1e-12)
    assert not S[0, 0, last + 1:].any()
    wts = rng.random(w)
    Sw = O.prefill_window_colsum(q, K, NL, Hq, Hkv, d, N, w, wts)
    parts = sum(wts[jj] * O.prefill_window_colsum(q, K, NL, Hq, Hkv, d, N, w, np.eye(w)[jj])
                for jj in range(w))
    np.testing.assert_allclose(Sw, parts, rtol=1e-12)


def test_ema_init_is_the_colsum_with_ema_weights():
    rng = np.random.default_rng(43)
    NL, Hq, Hkv, d, N, w, al = 1, 8, 2, 8, 30, 7, 0.8
    q = bf(rng.normal(size=(NL, Hq, w, d)))
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    wts = (1 - al) * al ** (w - 1 - np.arange(w))
    np.testing.assert_allclose(O.prefill_ema_init(q, K, NL, Hq, Hkv, d, N, w, al),
                               O.prefill_window_colsum(q, K, NL, Hq, Hkv, d, N, w, wts),
                               rtol=1e-14)


@pytest.mark.parametrize("N,pool", [(17, 4), (16, 4), (9, 1), (5, 8)])
def test_snapkv_block_means_and_sink(N, pool):
    """Blocks of `pool` consecutive positions take the mean of their tokens'
    accumulated attention (a ragged last block its own mean); the sink at
    position 0 scores +infinity; no sink leaves block 0 its mean."""
    rng = np.random.default_rng(44 + N)
    acc = rng.random((2, 3, N))
    s = O.snapkv_scores(acc, pool, sink=True)
    s0 = O.snapkv_scores(acc, pool, sink=False)
    for l, g in itertools.product(range(2), range(3)):
        for i in range(N):
            b = i // pool
            blk = acc[l, g, b * pool: min(N, (b + 1) * pool)]
            assert s0[l, g, i] == pytest.approx(blk.sum() / len(blk), rel=1e-15)
            if i > 0:
                assert s[l, g, i] == s0[l, g, i]
        assert s[l, g, 0] == math.inf


def test_snapkv_selection_keeps_sinks_and_splits_budgets_by_layer():
    """The protocol's selection: every layer keeps B_total / NL tokens over
    its KV heads (adaptive per-head budgets within the layer), the sink of
    every head first, then the highest pooled scores (brute-force sort)."""
    rng = np.random.default_rng(45)
    NL, Hq, Hkv, d, N, w, B = 2, 8, 2, 8, 40, 8, 24
    q = bf(rng.normal(size=(NL, Hq, w, d)))
    K = bf(rng.normal(size=(NL, Hkv, N, d)))
    res = O.prefill_snapkv(q, K, NL=NL, Hq=Hq, Hkv=Hkv, d=d, N=N, w=w, B_total=B)
    keep = res["keep"].astype(bool)
    assert keep.reshape(NL, -1).sum(axis=1).tolist() == [B // NL] * NL
    assert keep[:, :, 0].all()
    for l in range(NL):
        sc = res["scores"][l].ravel()
        order = sorted(range(sc.size), key=lambda j: (-sc[j], j))[: B // NL]
        assert sorted(order) == np.nonzero(keep[l].ravel())[0].tolist()
