"""GPU parity of the decode step (through the C ABI) against the fp64 oracle
on the seeded workloads: the small configurations in full, the large ones on
64 sampled units at full size and every step, plus edge cases."""
import numpy as np
import pytest
import torch

from kv_cache_eviction_kvc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from parity import run_decode_parity  # noqa: E402


def sample_units(U, n=64, seed=0):
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.arange(1, U - 1), size=n - 2, replace=False)
    return sorted({0, U - 1, *rest.tolist()})


def check(rep):
    print(rep)
    assert rep.ok(), rep


@pytest.mark.parametrize("fused", [True, False])
def test_c0_full(fused):
    check(run_decode_parity(W.C0, fused=fused))


def test_c1_full():
    check(run_decode_parity(W.C1))


def test_c2_sampled_full_size():
    check(run_decode_parity(W.C2, units=sample_units(W.C2.U)))


def test_c4_sampled_full_size():
    check(run_decode_parity(W.C4, units=sample_units(W.C4.U)))


SMALL = W.C0.with_(name="small", N=700, L=50, steps=24)


@pytest.mark.parametrize("cfg", [
    SMALL,                                                           # ragged chunk tail
    SMALL.with_(votes_max=8, rule=W.RULE_CUMULATIVE),
    SMALL.with_(rule=W.RULE_SINGLE, T=4),
    SMALL.with_(T=50, correction=W.CORR_ZERO_ORDER),                 # T = L
    SMALL.with_(correction=W.CORR_OFF, k_dist="mixture", centres=8),
    SMALL.with_(Hq=2, Hkv=2, N=300, L=20),                           # G = 1
    SMALL.with_(Hq=4, Hkv=2, N=129, L=128, steps=6),                 # k = 2 at step 1
    SMALL.with_(Hq=16, Hkv=2, B=2, N=513, L=17, votes_max=3),        # G = 8
    SMALL.with_(N=40, L=64, steps=30),                               # no eviction at first
    SMALL.with_(T=0),                                                # Score-Free
    SMALL.with_(N=100, L=100, T=0, steps=80),                        # queue of 70, then argmin
    SMALL.with_(Hq=8, Hkv=4, N=400, L=30),                           # G = 2 (first-step pass)
], ids=["ragged", "votes-cumulative", "single-lazy", "T=L-zero-order", "corr-off",
        "G1", "k2", "G8-votes", "under-budget", "score-free", "score-free-queue", "G2"])
@pytest.mark.parametrize("fused", [True, False])
def test_edge_cases(cfg, fused):
    check(run_decode_parity(cfg, fused=fused))


def test_device_status_reports_overlong_unit():
    from kv_cache_eviction_kvc_gb300.state import DecodeState
    cfg = SMALL
    st = DecodeState(2, 4, 80, 50, kmax=4)
    st.len.fill_(60)
    inp = W.gen_step(cfg, "cuda", 1)
    st.step(1, 60, inp["q"], inp["k_new"], inp["v_new"], max_len=55)   # 61 > 55
    torch.cuda.synchronize()
    assert st.device_status() == 2          # KVC_ERR_SHAPE recorded, nothing done
    assert st.len.tolist() == [60, 60]
    assert st.device_status() == 0          # reading clears it


@pytest.mark.parametrize("cfg", [
    SMALL.with_(merge_recent=8),                                     # KeepKV ZIP-merging
    SMALL.with_(Hq=2, Hkv=2, N=300, L=20, votes_max=4, merge_recent=0),   # G = 1, votes
    SMALL.with_(Hq=16, Hkv=2, B=2, N=513, L=17, merge_recent=3, T=4),     # G = 8, lazy
    SMALL.with_(N=40, L=32, steps=12, merge_recent=64),              # no candidate: evict
    SMALL.with_(merge_recent=8, T=4),                                # lazy: queue, search in pass 1
    SMALL.with_(Hq=4, Hkv=2, N=400, L=40, merge_recent=8, T=4),      # the same with G = 2
], ids=["zip", "zip-G1-votes", "zip-G8-lazy", "zip-no-candidate", "zip-G4-lazy", "zip-G2-lazy"])
@pytest.mark.parametrize("fused", [True, False])
def test_zip_merge(cfg, fused):
    rep = run_decode_parity(cfg, fused=fused)
    check(rep)
    if cfg.merge_recent < 64:
        assert rep.merges > 0


@pytest.mark.parametrize("fused", [True, False])
def test_zip_merge_c2_sampled_full_size(fused):
    rep = run_decode_parity(W.C2.with_(merge_recent=32), units=sample_units(W.C2.U), steps=24,
                            fused=fused)
    check(rep)
    assert rep.merges >= 64 * 22



@pytest.mark.parametrize("cfg", [
    SMALL.with_(rule=W.RULE_MI),                                     # 651 rounds at step 1
    SMALL.with_(rule=W.RULE_MI, Hq=2, Hkv=2, N=300, L=20, votes_max=4),   # G = 1, votes
    SMALL.with_(rule=W.RULE_MI, k_dist="mixture", centres=8, correction=W.CORR_ZERO_ORDER),
    SMALL.with_(rule=W.RULE_MI, Hq=16, Hkv=2, N=129, L=126, steps=8, votes_max=3),  # k = 4, G = 8
    W.C0.with_(rule=W.RULE_MI, steps=12),                            # the tiny workload, 449 rounds
], ids=["mi", "mi-G1-votes", "mi-mixture", "mi-k4-G8-votes", "mi-c0"])
@pytest.mark.parametrize("fused", [True, False])
def test_moment_informed(cfg, fused):
    """MomentKV's moment-aware phase: a first step removing several slots
    runs the loop of Algorithm 1 (kvc_mi_evict), later steps one round; the
    oracle replays the GPU's victims round by round."""
    rep = run_decode_parity(cfg, fused=fused)
    check(rep)
    assert rep.mi_rounds >= (cfg.N + 1 - cfg.L) * cfg.U


def test_moment_informed_c2_sampled_full_size():
    rep = run_decode_parity(W.C2_MI, units=sample_units(W.C2.U), steps=6)
    check(rep)
    assert rep.mi_rounds == 64 * 5


def test_aggregate_refuses_one_shot_moment_informed_eviction():
    """kvc_aggregate_evict under the moment-informed rule evicts one slot per
    unit; a unit that would lose several is refused on the device
    (KVC_ERR_UNSUPPORTED) and loses nothing: the loop is kvc_mi_evict's."""
    from kv_cache_eviction_kvc_gb300 import kvc as K
    from kv_cache_eviction_kvc_gb300.state import DecodeState
    cfg = SMALL.with_(N=60, L=50)
    st = DecodeState(2, 4, 80, 50, rule=W.RULE_MI, kmax=16)
    pre = W.gen_prefill(cfg.with_(B=1, NL=1, Hkv=2, Hq=8), "cuda", 0, cap=80)
    st.load_prefill(pre["K"], pre["V"], None, pre["pos"], pre["len"])
    inp = W.gen_step(cfg.with_(B=1, NL=1, Hkv=2, Hq=8), "cuda", 1)
    K.kvc_decode_attend(st.params, 1, 60, 61, inp["q"], inp["k_new"], inp["v_new"], st.cache,
                        st.lse, st.f_all, st.probs, st.ws)
    K.kvc_aggregate_evict(st.params, 1, st.probs, st.cache, st.kmax, st.evict_idx, st.evict_pos,
                          st.n_evict, st.ws)
    torch.cuda.synchronize()
    assert st.device_status() == 5
    assert st.n_evict.tolist() == [0, 0]


# ------------------------------------------- prefill selection -> hand-off -> decode

PIPE = W.C3.with_(name="pipe", NL=2, B_total=2 * 8 * 128)       # full prompt length, 2 layers


@pytest.mark.parametrize("scorer,rule,T,pc", [
    ("snapkv", W.RULE_EMA, 1, PIPE),                  # SnapKV protocol, EMA decode
    ("snapkv", W.RULE_MI, 1, PIPE),                   # MomentKV's pipeline: SnapKV then MI decode
    ("laprox", W.RULE_EMA, 4, PIPE),                  # LaProx global top-K, variable budgets, lazy
    ("laprox", W.RULE_EMA, 1, PIPE.with_(N=2000, B_total=40)),   # heads left empty: budget 1
], ids=["snapkv-ema", "snapkv-mi", "laprox-lazy", "laprox-empty-heads"])
def test_prefill_handoff_then_decode(scorer, rule, T, pc):
    """The prefill selection's kept set handed over to decoding: every unit
    keeps its own budget (LaProx key design 3; MomentKV's adaptive per-head
    allocation), the prompt's dropped tokens are the first eviction set of
    the moments (MomentKV Algorithm 1), and decode steps evict each unit
    down to its own budget."""
    from parity import run_pipeline_parity
    rep = run_pipeline_parity(pc, scorer=scorer, rule=rule, T=T, steps=10)
    print(rep)
    assert rep.ok(), rep
    assert rep.decode.steps == 10
    if scorer == "laprox":
        assert rep.min_kept != rep.max_kept            # budgets really vary


# ------------------------------------------------------ layer-chained EMA

@pytest.mark.parametrize("cfg", [
    W.C1.with_(rule=W.RULE_EMA_CHAINED, steps=24),                       # Llama-3.1-8B shape
    SMALL.with_(rule=W.RULE_EMA_CHAINED, B=2, NL=3, Hq=8, Hkv=2, N=300, L=40, T=4,
                votes_max=3),                                           # lazy, votes, 2 sequences
], ids=["chained-c1", "chained-lazy-votes"])
@pytest.mark.parametrize("fused", [True, False])
def test_layer_chained_ema(cfg, fused):
    """InertiaKV's evaluated aggregation: one EMA state per sequence passed
    through the layers in order; every unit of a sequence evicts the same
    positions (compared unit by unit against the oracle)."""
    check(run_decode_parity(cfg, fused=fused))
