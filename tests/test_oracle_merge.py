"""Pins of the oracle's KeepKV ZIP-merging against facts fixed outside it:
KeepKV Thm 3 (single-step lossless merge, checked with numpy attention), the
closed forms of eqs 10 and 12 at equal logits, the epsilon guard, brute-force
cosine candidate choice, and vote conservation over a whole generation.

Source: KeepKV reading notes (arXiv 2504.09936), "ZIP-Merging" eqs 6-13,
"why cosine similarity", "numerical stability" item 2, Algorithm 1.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def bf(x):
    return O.bf16_round(x)


def session(k, v, votes, G=1, cap=None, pos=None):
    n, d = k.shape
    s = O.DecodeSession(1, G, d, cap or n + 2)
    s.load(0, k, v, votes, pos)
    return s


def attention(qv, k, v, p):
    """Vote-weighted softmax attention of one query (KeepKV eq 6), numpy."""
    x = k @ qv / math.sqrt(k.shape[1])
    a = p * np.exp(x - x.max())
    return a @ v / a.sum(), math.log(a.sum()) + x.max()


def random_case(seed, n=12, d=16, G=1, vmax=4):
    rng = np.random.default_rng(seed)
    k = bf(rng.normal(size=(n, d)))
    v = bf(rng.normal(size=(n, d)))
    p = rng.integers(1, vmax + 1, size=n).astype(np.int32)
    q = bf(rng.normal(size=(1, G, d)))
    return k, v, p, q


def merged_cache(k, v, p, e, c, kr, vr):
    keep = [i for i in range(len(k)) if i not in (e, c)]
    k2 = np.vstack([k[keep], kr[None]])
    v2 = np.vstack([v[keep], vr[None]])
    p2 = np.append(p[keep], p[e] + p[c]).astype(float)
    return k2, v2, p2


@pytest.mark.parametrize("seed", range(8))
def test_theorem3_single_step_lossless(seed):
    """G = 1: attention over the merged cache (k_r, v_r, p_e + p_c replacing
    the pair) equals attention over the full cache, output and partition
    function, to rounding (KeepKV Thm 3, eq 13)."""
    k, v, p, q = random_case(seed)
    n = len(k)
    e = seed % n
    s = session(k, v, p)
    r = s.zip_merge(q, [e], new_pos=n, R=0)
    c = int(r["partner"][0])
    assert c >= 0 and c != e and r["guard"][0] == 0
    f_full, lz_full = attention(q[0, 0], k, v, p.astype(float))
    k2, v2, p2 = merged_cache(k, v, p, e, c, r["kr"][0], r["vr"][0])
    f_m, lz_m = attention(q[0, 0], k2, v2, p2)
    np.testing.assert_allclose(f_m, f_full, rtol=1e-11, atol=1e-12)
    assert lz_m == pytest.approx(lz_full, rel=1e-12)
    s.close()


@pytest.mark.parametrize("G", [2, 4, 8])
def test_theorem3_holds_for_the_group_mean_query(G):
    """GQA reading: the merge scores are the logits of the group's mean
    query, so Thm 3 holds exactly for that query (and not, in general, for
    each head)."""
    k, v, p, q = random_case(20 + G, G=G)
    s = session(k, v, p, G=G)
    e = 3
    r = s.zip_merge(q, [e], new_pos=len(k), R=0)
    c = int(r["partner"][0])
    k2, v2, p2 = merged_cache(k, v, p, e, c, r["kr"][0], r["vr"][0])
    qbar = q[0].mean(axis=0)
    f_full, _ = attention(qbar, k, v, p.astype(float))
    f_m, _ = attention(qbar, k2, v2, p2)
    np.testing.assert_allclose(f_m, f_full, rtol=1e-11, atol=1e-12)
    # a single head is not preserved exactly
    f_h, _ = attention(q[0, 0], k, v, p.astype(float))
    f_hm, _ = attention(q[0, 0], k2, v2, p2)
    assert np.abs(f_hm - f_h).max() > 1e-9
    s.close()


def test_equal_logits_give_vote_weighted_means():
    """Equal logits x_e = x_c = x: lambda = p / (p_e + p_c) and
    ell = ln((w_e + w_c)/(p_e + p_c)) = x, so eq 12 reduces to the
    vote-weighted mean key and eq 10 to the vote-weighted mean value."""
    d = 8
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((3, d))
    k[0] = [2, 1, 0, 0, 0, 0, 0, 0]       # victim
    k[1] = [2, -1, 3, 0, 0, 0, 0, 0]      # partner: same q . k, most similar
    k[2] = [-4, 0, 0, 0, 0, 0, 0, 1]
    v = bf(np.random.default_rng(3).normal(size=(3, d)))
    p = np.array([1, 3, 1], np.int32)
    s = session(k, v, p)
    r = s.zip_merge(q, [0], new_pos=3, R=0)
    assert r["partner"][0] == 1 and r["guard"][0] == 0
    np.testing.assert_allclose(r["kr"][0], (1 * k[0] + 3 * k[1]) / 4, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["vr"][0], (1 * v[0] + 3 * v[1]) / 4, rtol=1e-14, atol=1e-15)
    s.close()


def test_epsilon_guard_falls_back_to_the_plain_mean_key():
    """A query orthogonal to both keys gives a zero weighted mean logit: the
    key formula's denominator vanishes and the guard takes (k_e + k_c) / 2;
    the value is still the score-weighted mean (scores 1, so vote-weighted)."""
    d = 8
    q = np.zeros((1, 1, d)); q[0, 0, 7] = 1.0
    k = np.zeros((3, d))
    k[0] = [1, 2, 0, 0, 0, 0, 0, 0]
    k[1] = [1, 2.5, 0, 0, 0, 0, 0, 0]
    k[2] = [-1, 0, 1, 0, 0, 0, 0, 0]
    v = bf(np.random.default_rng(4).normal(size=(3, d)))
    p = np.array([2, 1, 1], np.int32)
    s = session(k, v, p)
    r = s.zip_merge(q, [0], new_pos=3, R=0)
    assert r["partner"][0] == 1 and r["guard"][0] == 1
    np.testing.assert_array_equal(r["kr"][0], (k[0] + k[1]) / 2)
    np.testing.assert_allclose(r["vr"][0], (2 * v[0] + v[1]) / 3, rtol=1e-14)
    s.close()


def brute_force_partner(k, pos, e, new_pos, R):
    best, arg = -np.inf, -1
    for i in sorted(range(len(k)), key=lambda i: pos[i]):
        if i == e or pos[i] > new_pos - R:
            continue
        ne, ni = np.linalg.norm(k[e]), np.linalg.norm(k[i])
        c = float(k[e] @ k[i] / (ne * ni)) if ne > 0 and ni > 0 else 0.0
        if c > best:
            best, arg = c, i
    return arg


@pytest.mark.parametrize("seed", range(10))
def test_partner_is_the_most_similar_older_key(seed):
    """Candidate choice against brute force: largest cosine of keys, the
    last R positions and the victim excluded, ties to the older token
    (duplicated keys force ties; a zero key has similarity 0)."""
    rng = np.random.default_rng(40 + seed)
    n, d = 14, 6
    k = bf(rng.integers(-2, 3, size=(n, d)).astype(float))
    k[rng.integers(0, n)] = 0.0
    dup = rng.choice(n, size=2, replace=False)
    k[dup[1]] = k[dup[0]]
    v = bf(rng.normal(size=(n, d)))
    pos = np.sort(rng.choice(100, size=n, replace=False)).astype(np.int32)
    new_pos = int(pos[-1])
    R = int(rng.integers(0, 6))
    e = int(rng.integers(0, n))
    q = bf(rng.normal(size=(1, 1, d)))
    s = session(k, v, np.ones(n, np.int32), pos=pos)
    r = s.zip_merge(q, [int(pos[e])], new_pos=new_pos, R=R)
    want = brute_force_partner(k, pos, e, new_pos, R)
    assert r["partner"][0] == (pos[want] if want >= 0 else -1)
    s.close()


def test_no_candidate_leaves_the_unit_untouched():
    """Every other slot within the last R positions: nothing is merged."""
    k, v, p, q = random_case(7, n=5)
    s = session(k, v, p)
    r = s.zip_merge(q, [0], new_pos=4, R=4)
    assert r["partner"][0] == -1
    n, pos, vote, _, _ = s.slots()
    assert n[0] == 5 and vote[0, :5].tolist() == p.tolist()
    s.close()


def test_bookkeeping_votes_utilities_positions():
    """After a merge the partner holds p_e + p_c, the sum of the two
    utilities, its own position and the bf16 rounding of (k_r, v_r); the
    victim's slot is gone and the others are unchanged."""
    k, v, p, q = random_case(9, n=6)
    s = session(k, v, p)
    probs = np.zeros((1, s.cap)); probs[0, :6] = [0.1, 0.2, 0.05, 0.3, 0.15, 0.2]
    s.update_util(probs, O.RULE_SINGLE, 0.0)
    r = s.zip_merge(q, [2], new_pos=6, R=0)
    c = int(r["partner"][0])
    n, pos, vote, util, _ = s.slots()
    assert n[0] == 5 and 2 not in pos[0, :5].tolist()
    j = pos[0, :5].tolist().index(c)
    assert vote[0, j] == p[2] + p[c]
    assert util[0, j] == pytest.approx(probs[0, 2] + probs[0, c], rel=1e-15)
    K, V = s.rows()
    np.testing.assert_array_equal(O.bf16_round(r["kr"][0]), _b2f(K[0, j]))
    np.testing.assert_array_equal(O.bf16_round(r["vr"][0]), _b2f(V[0, j]))
    for i in range(5):
        if i != j:
            src = pos[0, i]
            np.testing.assert_array_equal(_b2f(K[0, i]), k[src])
    s.close()


def _b2f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_generation_conserves_votes_and_matches_full_attention():
    """Whole decode loop in merge mode: every token's vote is either in the
    cache or in the eviction moments (sum of votes + n_e = tokens seen), a
    merging step leaves the moments unchanged, and its output is the
    attention over the cache before the merge (numpy, from the step's
    inputs and the previous step's rows)."""
    rng = np.random.default_rng(17)
    U, N, d, G, S, L = 2, 20, 8, 2, 10, 9
    kp, vp = bf(rng.normal(size=(U, N, d))), bf(rng.normal(size=(U, N, d)))
    qs = bf(rng.normal(size=(S, U, G, d)))
    ks, vs = bf(rng.normal(size=(S, U, d))), bf(rng.normal(size=(S, U, d)))
    sess = O.DecodeSession(U, G, d, N + S)
    for u in range(U):
        sess.load(u, kp[u], vp[u])
    prev_ne = None
    n_merged = 0
    for s_ in range(S):
        t = s_ + 1
        n0, pos0, vote0, _, _ = sess.slots()
        K0, V0 = sess.rows()
        r = O.decode_step(sess, t, N + t - 1, qs[s_], ks[s_], vs[s_], L=L, rule=O.RULE_EMA,
                          alpha=0.9, T=1, correction=O.CORR_OFF, merge_recent=2)
        n, _, vote, _, _ = sess.slots()
        ne = sess.moments()[0]
        assert (n == L).all()
        for u in range(U):
            assert vote[u, :n[u]].sum() + ne[u] == N + t
            if t > 1 and r["merged"][u]:
                n_merged += 1
                assert ne[u] == prev_ne[u]
                kk = np.vstack([_b2f(K0[u, :n0[u]]), ks[s_, u]])
                vv = np.vstack([_b2f(V0[u, :n0[u]]), vs[s_, u]])
                pp = np.append(vote0[u, :n0[u]], 1).astype(float)
                for h in range(G):
                    f, _ = attention(qs[s_, u, h], kk, vv, pp)
                    np.testing.assert_allclose(r["o"][u, h], f, rtol=1e-10, atol=1e-12)
        assert not r["merged"].any() if t == 1 else True
        prev_ne = ne
    assert n_merged >= S - 3
    sess.close()


def test_figure3_worked_votes():
    """The worked merge of the KeepKV notes' Figure 3 (tests/golden): votes
    1 and 2 merge into one entry of vote 3 with weights 1 s_e and 2 s_c, and
    the output over the merged cache equals the output before (Thm 3)."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "keepkv_fig3_merge.json")))
    rng = np.random.default_rng(77)
    d = 16
    k = bf(rng.normal(size=(4, d)))
    v = bf(rng.normal(size=(4, d)))
    k[1] = bf(k[0] + 0.05 * rng.normal(size=d))      # slot 1: the victim's most similar key
    p = np.array([g["p_e"], g["p_c"], 1, 1], np.int32)
    q = bf(rng.normal(size=(1, 1, d)))
    s = session(k, v, p)
    r = s.zip_merge(q, [0], new_pos=4, R=0)
    assert int(r["partner"][0]) == 1
    _, _, vote, _, _ = s.slots()
    assert sorted(vote[0, :3].tolist()) == sorted([g["p_r"], 1, 1])
    # v_r = (w_e v_e + w_c v_c) / (w_e + w_c) with w = (vote) * s and s = exp(q k / sqrt(d))
    se = math.exp(float(k[0] @ q[0, 0]) / math.sqrt(d))
    sc = math.exp(float(k[1] @ q[0, 0]) / math.sqrt(d))
    we, wc = g["w_e_over_s_e"] * se, g["w_c_over_s_c"] * sc
    np.testing.assert_allclose(r["vr"][0], (we * v[0] + wc * v[1]) / (we + wc), rtol=1e-12)
    f_full, _ = attention(q[0, 0], k, v, p.astype(float))
    k2, v2, p2 = merged_cache(k, v, p, 0, 1, r["kr"][0], r["vr"][0])
    f_m, _ = attention(q[0, 0], k2, v2, p2)
    np.testing.assert_allclose(f_m, f_full, rtol=1e-11, atol=1e-12)
    s.close()
