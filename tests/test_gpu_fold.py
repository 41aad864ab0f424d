"""The eviction-set moment fold with many victims per unit (the tensor-core
kernel kvc_moment_update takes from 256 victims per unit on) against the
oracle's fold (MomentKV sec 4.1: n, mu_k, mu_v, C = S~ / n of the evicted
tokens; KeepKV votes as weights).  Two folds in a row, so the second merges
into non-zero moments; ragged tile tails; a unit with no victims; keys and
values with means several spreads away from zero (the centring the kernel
does per 128-victim tile has to hold there); votes above 256 (w v no longer
exact in two bf16 terms)."""
import numpy as np
import pytest
import torch

from kv_cache_eviction_kvc_gb300 import kvc as K
from kv_cache_eviction_kvc_gb300.state import DecodeState
from oracle import oracle as O
from parity import MOM_TOL, _rel

pytestmark = pytest.mark.gpu


def _case(seed, U, n, votes_max, offset):
    rng = np.random.default_rng(seed)
    d = 128
    k = O.bf16_round(offset[0] + rng.standard_normal((U, n, d)) * 1.0)
    v = O.bf16_round(offset[1] + rng.standard_normal((U, n, d)) * 0.5)
    vote = rng.integers(1, votes_max + 1, (U, n)).astype(np.int32) if votes_max else None
    return rng, k, v, vote


@pytest.mark.parametrize("votes_max,offset,ks", [
    (0, (0.0, 0.0), ((300, 0, 1000), (777, 513, 129))),
    (0, (3.0, -2.0), ((640, 257, 999), (512, 300, 1))),
    (8, (1.5, 0.5), ((449, 1000, 0), (1100, 256, 700))),
    (300, (0.0, 1.0), ((384, 385, 383), (260, 900, 1030))),
])
def test_fold_matches_oracle(votes_max, offset, ks):
    U, n, G, d = 3, 2200, 4, 128
    rng, k, v, vote = _case(17 + votes_max, U, n, votes_max, offset)
    dev = torch.device("cuda", 0)
    st = DecodeState(U, G, n + 8, n, votes=vote is not None, device=dev)
    kt = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16).to(dev)
    vt = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(dev)
    vo = None if vote is None else torch.from_numpy(vote).to(dev)
    pos = torch.arange(n, dtype=torch.int32, device=dev).repeat(U, 1)
    st.load_prefill(kt, vt, vo, pos, torch.full((U,), n, dtype=torch.int32, device=dev))
    sess = O.DecodeSession(U, G, d, n + 8)
    for u in range(U):
        sess.load(u, k[u], v[u], None if vote is None else vote[u], np.arange(n, dtype=np.int32))
    # two disjoint victim batches per unit
    perm = [rng.permutation(n) for _ in range(U)]
    used = [0] * U
    for batch in ks:
        kmax = max(max(batch), 1)
        vic = np.full((U, kmax), -1, np.int32)
        nv = np.zeros(U, np.int32)
        for u in range(U):
            c = batch[u]
            vic[u, :c] = np.sort(perm[u][used[u]:used[u] + c])
            nv[u] = c
            used[u] += c
        ev = torch.from_numpy(vic).to(dev)
        ne = torch.from_numpy(nv).to(dev)
        K.kvc_moment_update(st.params, st.cache, kmax, ev, ne, st.moments, st.ws)
        sess.evict(vic, nv)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    n_r, mk_r, mv_r, C_r = sess.moments()
    n_g = st.n.cpu().numpy().astype(np.float64)
    mk_g = st.mu_k.cpu().numpy().astype(np.float64)
    mv_g = st.mu_v.cpu().numpy().astype(np.float64)
    C_g = st.C.cpu().numpy().astype(np.float64)
    sess.close()
    np.testing.assert_array_equal(n_g, n_r)
    for u in range(U):
        assert _rel(mk_g[u], mk_r[u]) <= MOM_TOL, (u, _rel(mk_g[u], mk_r[u]))
        assert _rel(mv_g[u], mv_r[u]) <= MOM_TOL, (u, _rel(mv_g[u], mv_r[u]))
        assert _rel(C_g[u], C_r[u]) <= MOM_TOL, (u, _rel(C_g[u], C_r[u]))
