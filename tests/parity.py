"""GPU-vs-oracle parity driver for the decode step (test helper).

The CUDA path (through the C ABI) and the fp64 oracle run the same seeded
inputs step by step.  Each step compares:

* eviction sets, by token position: they must be equal, except that a token
  in the symmetric difference is accepted when the oracle's utility for it is
  within 1e-6 relative of the oracle's k-th (threshold) utility (a near-tie:
  both choices are valid orders of equal-up-to-rounding utilities).  Accepted
  near-tie choices are counted; the oracle then applies the GPU's set, which
  is one of the valid sets, so one tie does not change every later step.
  Any other difference is a mismatch (the test fails).
* the corrected output o: max over units and heads of
  ||o_gpu - o_ref||_inf / ||o_ref||_inf <= 2e-3;
* the moments: ||d mu|| / ||mu|| and ||d C||_F / ||C||_F <= 1e-4 per unit
  (absolute 1e-6 when the norm is below 1e-3), n exact;
* the head-mean probabilities on refresh steps (by position), and with the
  five-call path lse and f_all;
* in ZIP-merge mode (KeepKV), the partner of each merged victim: the oracle
  merges into the GPU's partner when that partner's key cosine is within
  1e-5 of the best one (counted as a near-tie when below it), otherwise the
  step is a mismatch; the merged key and value rows must be within one bf16
  unit of the oracle's unrounded k_r, v_r (either guard branch is accepted
  when the weighted mean logit is within 0.1 % of the guard threshold), and
  the oracle then adopts the GPU's rows;
* under MomentKV's moment-informed rule, the step's scores alpha ||r|| (the
  utilities of the retained slots, by position) within 2e-3 relative (floor:
  1e-4 of the unit's largest score); the oracle replays the GPU's victims
  round by round (MomentKV Algorithm 1 removes one slot per round and
  re-scores), and each must score within 1e-4 of that round's lowest score
  (the scores are functions of the moments, whose tolerance is 1e-4).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from kv_cache_eviction_kvc_gb300 import workloads as W
from kv_cache_eviction_kvc_gb300.state import DecodeState
from oracle import oracle as O

TIE_REL = 1e-6
O_TOL = 2e-3
MOM_TOL = 1e-4
PROB_TOL = 2e-3   # head-mean probabilities are attention outputs
COS_BAND = 1e-5   # partner near-tie band (key cosines, fp32 on the GPU)
MI_TIE_REL = 1e-4     # near-tie band of moment-informed scores
MI_SCORE_TOL = 2e-3
ROW_REL = 2.0 ** -7   # one bf16 unit (8 significand bits)


@dataclasses.dataclass
class ParityReport:
    steps: int = 0
    band_hits: int = 0
    mismatches: int = 0
    max_o_err: float = 0.0
    max_mu_err: float = 0.0
    max_C_err: float = 0.0
    max_prob_err: float = 0.0
    max_lse_err: float = 0.0
    max_fall_err: float = 0.0
    n_err: int = 0
    merges: int = 0
    max_row_err: float = 0.0      # merged rows, in bf16 units of the reference
    max_mi_err: float = 0.0       # moment-informed scores (retained slots)
    mi_rounds: int = 0            # moment-aware eviction rounds compared
    max_mi_gap: float = 0.0       # largest accepted relative score gap of a round
    first_mismatch: str = ""

    def ok(self):
        return (self.mismatches == 0 and self.max_o_err <= O_TOL and self.max_mu_err <= MOM_TOL
                and self.max_C_err <= MOM_TOL and self.max_prob_err <= PROB_TOL
                and self.n_err == 0 and self.max_lse_err <= O_TOL and self.max_fall_err <= O_TOL
                and self.max_mi_err <= MI_SCORE_TOL)


def _rel(a, b, floor=1e-3, absfloor=1e-6):
    nb = np.linalg.norm(b)
    d = np.linalg.norm(a - b)
    return d / nb if nb >= floor else (0.0 if d <= absfloor else d / max(nb, 1e-30))


def run_decode_parity(cfg: W.DecodeConfig, *, steps: int | None = None, units=None,
                      fused: bool = True, seed: int = 0, device="cuda",
                      cap: int | None = None) -> ParityReport:
    S = cfg.steps if steps is None else steps
    merge = cfg.merge_recent is not None
    U, G, d, N, L = cfg.U, cfg.G, cfg.d, cfg.N, cfg.L
    units = list(range(U)) if units is None else list(units)
    uidx = torch.tensor(units, device=device, dtype=torch.long)
    cap = max(N + 1, L + 1) if cap is None else cap
    P = W.unit_params(cfg, device, seed)
    pre = W.gen_prefill(cfg, device, seed, cap=cap, P=P)
    chained = cfg.rule == W.RULE_EMA_CHAINED
    if chained:
        assert len(units) == U, "the layer-chained EMA compares whole sequences"
    st = DecodeState(U, G, cap, L, rule=cfg.rule, alpha=cfg.alpha, refresh_period=cfg.T,
                     correction=cfg.correction, votes=bool(cfg.votes_max) or merge,
                     kmax=max(1, N + 1 - L), device=device, merge_recent=cfg.merge_recent,
                     chain=(cfg.NL, cfg.Hkv) if chained else None)
    st.load_prefill(pre["K"], pre["V"], pre["votes"], pre["pos"], pre["len"])
    sess = O.DecodeSession(len(units), G, d, cap + 1)
    Kh = pre["K"][uidx, :N].cpu()
    Vh = pre["V"][uidx, :N].cpu()
    vh = None if pre["votes"] is None else pre["votes"][uidx, :N].cpu().numpy()
    for j in range(len(units)):
        sess.load(j, Kh[j], Vh[j], None if vh is None else vh[j], np.arange(N, dtype=np.int32))
    del Kh, Vh, pre
    rep = ParityReport()
    try:
        _step_loop(cfg, st, sess, units, uidx, P, seed, device, fused, S, N, L, rep)
    finally:
        sess.close()
    return rep


def _step_loop(cfg, st, sess, units, uidx, P, seed, device, fused, S, n_len, L, rep):
    """Steps 1..S of the decode stream on the GPU state ``st`` and the oracle
    session ``sess`` (units ``units`` of the GPU state), compared step by step
    into ``rep``.  L: one budget, or one per compared unit."""
    N = cfg.N
    merge = cfg.merge_recent is not None
    for t in range(1, S + 1):
        inp = W.gen_step(cfg, device, t, seed, P)
        new_pos = N + t - 1
        max_len = n_len + 1
        rule = cfg.first_rule if (t == 1 and cfg.first_rule is not None) else cfg.rule
        mi = rule == W.RULE_MI
        tie_rel = MI_TIE_REL if mi else TIE_REL
        st.params.rule = rule
        refresh = True if mi else O.is_refresh(t, cfg.T)
        pos_before = st.pos[uidx, :max_len].cpu().numpy().copy()
        votes_before = st.votes[uidx, :max_len].cpu().numpy().copy() if merge else None
        len_before = st.len[uidx].cpu().numpy().copy()
        if fused:
            st.step(t, new_pos, inp["q"], inp["k_new"], inp["v_new"], max_len)
        else:
            st.step_calls(t, new_pos, inp["q"], inp["k_new"], inp["v_new"], max_len)
        torch.cuda.synchronize()
        ds = st.device_status()
        assert ds == 0, f"device status {ds} at step {t}"
        nev = st.n_evict[uidx].cpu().numpy()
        partner_g = None
        if merge and not fused:
            partner_g = st.partner_pos[uidx].cpu().numpy()
        elif merge:
            # kvc_decode_step reports no partner: it is the one slot whose
            # vote grew (a merge adds the victim's vote to the partner's)
            partner_g = _partners_from_votes(new_pos, len_before, pos_before, votes_before,
                                             st.len[uidx].cpu().numpy(),
                                             st.pos[uidx].cpu().numpy(),
                                             st.votes[uidx].cpu().numpy())
        if merge:
            nev = nev + (partner_g >= 0)          # a merged victim left n_evict at 0
        evp = st.evict_pos[uidx].cpu().numpy()
        o_gpu = st.o[uidx].cpu().numpy().astype(np.float64)
        probs_gpu = st.probs[uidx, :max_len].cpu().numpy() if refresh else None
        if not fused:
            lse_gpu = st.lse[uidx].cpu().numpy()
            fall_gpu = st.f_all[uidx].cpu().numpy()

        qh = inp["q"][uidx].cpu()
        kh = inp["k_new"][uidx].cpu()
        vh2 = inp["v_new"][uidx].cpu()

        def choose(tt, prop):
            nonlocal rep
            n_o, pos_o, _, util_o, _ = sess.slots()
            vic, nv, thr = prop["victims"], prop["nvict"], prop["thr"]
            kmax = max(1, int(nev.max()), vic.shape[1])
            out = np.full((len(units), kmax), -1, np.int32)
            for j in range(len(units)):
                g = set(evp[j, : nev[j]].tolist())
                o_set = set(vic[j, : nv[j]].tolist())
                if g != o_set:
                    umap = dict(zip(pos_o[j, : n_o[j]].tolist(), util_o[j, : n_o[j]].tolist()))
                    bad = [p for p in g ^ o_set
                           if p not in umap or abs(umap[p] - thr[j]) > tie_rel * abs(thr[j])]
                    if bad or len(g) != len(o_set):
                        rep.mismatches += 1
                        if not rep.first_mismatch:
                            rep.first_mismatch = (f"step {tt} unit {units[j]}: gpu-only "
                                                  f"{sorted(g - o_set)[:5]} oracle-only "
                                                  f"{sorted(o_set - g)[:5]} thr {thr[j]!r}")
                    else:
                        rep.band_hits += 1
                gl = sorted(g)
                out[j, : len(gl)] = gl
            return out, nev.astype(np.int32)

        mi_forced = None
        if mi:
            # the GPU's victims in eviction order, replayed round by round
            kf = max(1, int(nev.max()))
            mi_forced = np.full((len(units), kf), -1, np.int32)
            for j in range(len(units)):
                mi_forced[j, : nev[j]] = evp[j, : nev[j]]
        try:
            prop = O.decode_step(sess, t, new_pos, qh, kh, vh2, L=L, rule=rule,
                                 alpha=cfg.alpha, T=cfg.T, correction=cfg.correction,
                                 choose=None if mi else choose,
                                 merge_recent=cfg.merge_recent,
                                 force_partner=partner_g, mi_forced=mi_forced,
                                 chain=(cfg.NL, cfg.Hkv))
        except ValueError as ex:
            rep.mismatches += 1
            rep.first_mismatch = rep.first_mismatch or f"step {t}: oracle refused: {ex}"
            break
        if mi:
            for j in range(len(units)):
                if prop["nvict"][j] != nev[j]:
                    rep.mismatches += 1
                    rep.first_mismatch = rep.first_mismatch or (
                        f"step {t} unit {units[j]}: gpu removed {nev[j]}, "
                        f"oracle {prop['nvict'][j]}")
                    continue
                for r in range(int(nev[j])):
                    b_, u_ = prop["mi_best"][j, r], prop["mi_used"][j, r]
                    rep.mi_rounds += 1
                    gap = (u_ - b_) / max(abs(b_), 1e-300)
                    if gap > MI_TIE_REL:
                        rep.mismatches += 1
                        rep.first_mismatch = rep.first_mismatch or (
                            f"step {t} unit {units[j]} round {r}: gpu victim "
                            f"{mi_forced[j, r]} scores {u_!r}, the lowest is {b_!r}")
                    elif gap > 0:
                        rep.band_hits += 1
                        rep.max_mi_gap = max(rep.max_mi_gap, float(gap))
        if merge:
            _check_merge(rep, t, units, st, uidx, sess, prop, partner_g)
        # output
        o_ref = prop["o"]
        num = np.abs(o_gpu - o_ref).max(axis=2)
        den = np.abs(o_ref).max(axis=2)
        rep.max_o_err = max(rep.max_o_err, float((num / np.maximum(den, 1e-30)).max()))
        if not fused:
            rep.max_lse_err = max(rep.max_lse_err, float(np.abs(lse_gpu - prop["lse"]).max()))
            fn = np.abs(fall_gpu - prop["f_all"]).max(axis=2)
            fd = np.abs(prop["f_all"]).max(axis=2)
            rep.max_fall_err = max(rep.max_fall_err, float((fn / np.maximum(fd, 1e-30)).max()))
        if refresh:
            pr = prop["probs"]
            for j in range(len(units)):
                nb = int(len_before[j])
                gp = probs_gpu[j, : nb + 1]
                gpos = np.append(pos_before[j, :nb], new_pos)
                order = np.argsort(gpos)
                ref = pr[j, : nb + 1]          # oracle slots are in position order
                err = np.abs(gp[order] - ref) / np.maximum(ref, 1e-300)
                rep.max_prob_err = max(rep.max_prob_err, float(err.max()))
        if mi:
            # the step's scores are the utilities of every retained slot
            ng_, pg_, ug_ = (st.len[uidx].cpu().numpy(), st.pos[uidx].cpu().numpy(),
                             st.util[uidx].cpu().numpy())
            no_, po_, _, uo_, _ = sess.slots()
            for j in range(len(units)):
                ref = dict(zip(po_[j, : no_[j]].tolist(), uo_[j, : no_[j]].tolist()))
                floor = 1e-4 * max(ref.values()) if ref else 0.0
                for p_, g_ in zip(pg_[j, : ng_[j]].tolist(), ug_[j, : ng_[j]].tolist()):
                    r_ = ref[p_]
                    rep.max_mi_err = max(rep.max_mi_err, abs(g_ - r_) / max(abs(r_), floor, 1e-300))
        # moments
        n_g = st.n[uidx].cpu().numpy()
        mk_g = st.mu_k[uidx].cpu().numpy()
        mv_g = st.mu_v[uidx].cpu().numpy()
        C_g = st.C[uidx].cpu().numpy()
        n_r, mk_r, mv_r, C_r = sess.moments()
        rep.n_err += int((n_g != n_r).sum())
        for j in range(len(units)):
            rep.max_mu_err = max(rep.max_mu_err, _rel(mk_g[j], mk_r[j]), _rel(mv_g[j], mv_r[j]))
            rep.max_C_err = max(rep.max_C_err, _rel(C_g[j], C_r[j]))
        n_len = int(st.len.max().item())
        st.params.rule = cfg.rule
        rep.steps += 1


def _partners_from_votes(new_pos, len0, pos0, votes0, len1, pos1, votes1):
    out = np.full(len(len0), -1, np.int32)
    for j in range(len(len0)):
        before = dict(zip(pos0[j, : len0[j]].tolist(), votes0[j, : len0[j]].tolist()))
        before[new_pos] = 1                   # the step's token (a partner when R = 0)
        grew = [p for p, v in zip(pos1[j, : len1[j]].tolist(), votes1[j, : len1[j]].tolist())
                if p in before and v > before[p]]
        if len(grew) == 1:
            out[j] = grew[0]
        elif len(grew) > 1:
            raise AssertionError(f"unit {j}: several votes grew {grew[:4]}")
    return out


def _check_merge(rep, t, units, st, uidx, sess, prop, partner_g):
    """Partner choice and merged rows of one merge-mode step (see the module
    docstring); the oracle adopts the GPU's merged rows."""
    mres, merged = prop["merge"], prop["merged"]
    pos_g = st.pos[uidx].cpu().numpy()
    for j in range(len(units)):
        g_m = partner_g[j] >= 0
        if g_m != bool(merged[j]):
            rep.mismatches += 1
            rep.first_mismatch = rep.first_mismatch or (
                f"step {t} unit {units[j]}: gpu merged {g_m} oracle merged {bool(merged[j])}")
            continue
        if not g_m:
            continue
        rep.merges += 1
        gap = mres["cos_best"][j] - mres["cos_used"][j]
        if gap > COS_BAND:
            rep.mismatches += 1
            rep.first_mismatch = rep.first_mismatch or (
                f"step {t} unit {units[j]}: partner {partner_g[j]} cosine {gap!r} below the best")
            continue
        if gap > 0:
            rep.band_hits += 1
        slot = int(np.nonzero(pos_g[j] == partner_g[j])[0][0])
        kb = st.K[units[j], slot].cpu().view(torch.int16).numpy().view(np.uint16)
        vb = st.V[units[j], slot].cpu().view(torch.int16).numpy().view(np.uint16)
        kg = (kb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        vg = (vb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        err = 0.0
        for g_, r_ in ((kg, mres["kr"][j]), (vg, mres["vr"][j])):
            e_ = np.abs(g_ - r_) / (ROW_REL * np.abs(r_) + 1e-6)
            err = max(err, float(e_.max()))
        if err > 1.0:
            near = abs(abs(mres["xt"][j]) - O.ZIP_EPS) <= 1e-3 * O.ZIP_EPS
            if near:
                rep.band_hits += 1
            else:
                rep.mismatches += 1
                rep.first_mismatch = rep.first_mismatch or (
                    f"step {t} unit {units[j]}: merged row off by {err:.2f} bf16 units "
                    f"(guard {mres['guard'][j]}, xt {mres['xt'][j]!r})")
        else:
            rep.max_row_err = max(rep.max_row_err, err)
        sess.set_row(j, int(partner_g[j]), kb, vb)


# ---------------------------------------------------------------------------
# prefill scorer
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class PrefillReport:
    band_hits: int = 0
    mismatches: int = 0
    max_gram_err: float = 0.0      # of R^T R against the oracle's Gram
    max_s_err: float = 0.0
    counts_ok: bool = True
    idx_ok: bool = True
    kept: int = 0
    first_mismatch: str = ""

    def ok(self):
        return (self.mismatches == 0 and self.max_gram_err <= MOM_TOL
                and self.max_s_err <= O_TOL and self.counts_ok and self.idx_ok)


def run_prefill_parity(cfg: W.PrefillConfig, *, seed: int = 0, device="cuda",
                       normalize: bool = True, alloc: int = 0) -> PrefillReport:
    """alloc: 0 global top-K (LaProx), 1 per layer (head-flatten only),
    2 uniform per KV head; near-ties are measured against the threshold of
    the element's own segment."""
    from kv_cache_eviction_kvc_gb300 import kvc as K
    NL, Hq, Hkv, d, N, w, B = cfg.NL, cfg.Hq, cfg.Hkv, cfg.d, cfg.N, cfg.w, cfg.B_total
    inp = W.gen_prefill_scorer(cfg, device, seed)
    R = torch.empty(NL, Hkv, d, d, dtype=torch.float32, device=device)
    K.kvc_prefill_prepare(NL, Hq, Hkv, d, cfg.D, inp["W_O"], R)
    M = NL * Hkv * N
    ws = torch.empty(max(256, K.kvc_prefill_workspace_size(NL, Hkv, N, B)), dtype=torch.uint8,
                     device=device)
    scores = torch.empty(NL, Hkv, N, dtype=torch.float32, device=device)
    keep = torch.empty(NL, Hkv, N, dtype=torch.uint8, device=device)
    counts = torch.empty(NL, Hkv, dtype=torch.int32, device=device)
    idx = torch.empty(max(B, 1), dtype=torch.int64, device=device)
    K.kvc_prefill_score(NL, Hq, Hkv, d, N, w, B, int(normalize), inp["q_win"], inp["K"],
                        inp["V"], R, scores, keep, counts, idx, ws, alloc=alloc)
    torch.cuda.synchronize()
    ref = O.prefill_score(inp["q_win"], inp["K"], inp["V"], inp["W_O"], NL=NL, Hq=Hq, Hkv=Hkv,
                          d=d, N=N, w=w, B_total=B, normalize=normalize, alloc=alloc)
    rep = PrefillReport()
    # the factor is not unique; R^T R is the Gram matrix
    Rn = R.cpu().numpy().astype(np.float64)
    g = np.einsum("lgka,lgkb->lgab", Rn, Rn)
    rep.max_gram_err = float(np.abs(g - ref["Gram"]).max() / np.abs(ref["Gram"]).max())
    s_gpu = scores.cpu().numpy().astype(np.float64)
    s_ref = ref["s"]
    rep.max_s_err = float((np.abs(s_gpu - s_ref) / np.maximum(np.abs(s_ref), 1e-30)).max())
    kg = keep.cpu().numpy().astype(bool).ravel()
    kr = ref["keep"].astype(bool).ravel()
    diff = np.nonzero(kg ^ kr)[0]
    thr = np.atleast_1d(ref["thr"])
    seg = M // len(thr)
    flat_s = s_ref.ravel()
    for j in diff:
        t_ = thr[j // seg]
        if abs(flat_s[j] - t_) <= TIE_REL * abs(t_):
            rep.band_hits += 1
        else:
            rep.mismatches += 1
            if not rep.first_mismatch:
                rep.first_mismatch = f"flat {j}: s_ref {flat_s[j]!r} thr {t_!r} gpu keep {kg[j]}"
    rep.kept = int(kg.sum())
    rep.counts_ok = bool(rep.kept == B and np.array_equal(
        counts.cpu().numpy(), kg.reshape(NL, Hkv, N).sum(axis=2)))
    rep.idx_ok = bool(np.array_equal(idx[:B].cpu().numpy(), np.nonzero(kg)[0]))
    return rep


# ---------------------------------------------------------------------------
# window attention column sums and MomentKV's SnapKV prefill protocol
# ---------------------------------------------------------------------------

def run_window_parity(cfg: W.PrefillConfig, weights, *, seed: int = 0, device="cuda") -> float:
    """Largest relative error of kvc_prefill_window_attention's weighted
    column sums against the oracle (relative to each element, floor 1e-6 of
    the (layer, KV head)'s largest)."""
    from kv_cache_eviction_kvc_gb300 import kvc as K
    NL, Hq, Hkv, d, N, w = cfg.NL, cfg.Hq, cfg.Hkv, cfg.d, cfg.N, cfg.w
    inp = W.gen_prefill_scorer(cfg, device, seed)
    ws = torch.empty(K.kvc_prefill_workspace_size(NL, Hkv, N, 0), dtype=torch.uint8, device=device)
    S = torch.empty(NL, Hkv, N, dtype=torch.float32, device=device)
    K.kvc_prefill_window_attention(NL, Hq, Hkv, d, N, w, list(weights), inp["q_win"], inp["K"], S,
                                   ws)
    torch.cuda.synchronize()
    ref = O.prefill_window_colsum(inp["q_win"], inp["K"], NL, Hq, Hkv, d, N, w,
                                  np.asarray(weights, dtype=np.float64))
    g = S.cpu().numpy().astype(np.float64)
    floor = 1e-6 * np.abs(ref).max(axis=2, keepdims=True)
    return float((np.abs(g - ref) / np.maximum(np.abs(ref), np.maximum(floor, 1e-30))).max())


def run_snapkv_parity(cfg: W.PrefillConfig, *, pool: int = 4, sink: bool = True, seed: int = 0,
                      device="cuda") -> PrefillReport:
    """kvc_prefill_snapkv against the oracle's protocol: scores per element
    (finite ones), the keep set exact outside the 1e-6 band around each
    layer's threshold, counts and the ascending per-layer index slices."""
    from kv_cache_eviction_kvc_gb300 import kvc as K
    NL, Hq, Hkv, d, N, w, B = cfg.NL, cfg.Hq, cfg.Hkv, cfg.d, cfg.N, cfg.w, cfg.B_total
    inp = W.gen_prefill_scorer(cfg, device, seed)
    ws = torch.empty(K.kvc_prefill_workspace_size(NL, Hkv, N, B), dtype=torch.uint8, device=device)
    scores = torch.empty(NL, Hkv, N, dtype=torch.float32, device=device)
    keep = torch.empty(NL, Hkv, N, dtype=torch.uint8, device=device)
    counts = torch.empty(NL, Hkv, dtype=torch.int32, device=device)
    idx = torch.empty(max(B, 1), dtype=torch.int64, device=device)
    K.kvc_prefill_snapkv(NL, Hq, Hkv, d, N, w, B, pool, int(sink), inp["q_win"], inp["K"], scores,
                         keep, counts, idx, ws)
    torch.cuda.synchronize()
    ref = O.prefill_snapkv(inp["q_win"], inp["K"], NL=NL, Hq=Hq, Hkv=Hkv, d=d, N=N, w=w,
                           B_total=B, pool=pool, sink=sink)
    rep = PrefillReport()
    s_gpu = scores.cpu().numpy().astype(np.float64)
    s_ref = ref["scores"]
    fin = np.isfinite(s_ref)
    if not np.array_equal(fin, np.isfinite(s_gpu)):
        rep.mismatches += 1
        rep.first_mismatch = "sink positions differ"
    rep.max_s_err = float((np.abs(s_gpu[fin] - s_ref[fin]) / np.maximum(np.abs(s_ref[fin]), 1e-30)).max())
    kg = keep.cpu().numpy().astype(bool).ravel()
    kr = ref["keep"].astype(bool).ravel()
    thr = np.atleast_1d(ref["thr"])
    seg = NL * Hkv * N // len(thr)
    flat_s = s_ref.ravel()
    for j in np.nonzero(kg ^ kr)[0]:
        t_ = thr[j // seg]
        if np.isfinite(flat_s[j]) and abs(flat_s[j] - t_) <= TIE_REL * abs(t_):
            rep.band_hits += 1
        else:
            rep.mismatches += 1
            if not rep.first_mismatch:
                rep.first_mismatch = f"flat {j}: s_ref {flat_s[j]!r} thr {t_!r} gpu keep {kg[j]}"
    rep.kept = int(kg.sum())
    rep.counts_ok = bool(rep.kept == B and np.array_equal(
        counts.cpu().numpy(), kg.reshape(NL, Hkv, N).sum(axis=2)))
    rep.idx_ok = bool(np.array_equal(idx[:B].cpu().numpy(), np.nonzero(kg)[0]))
    return rep



# ---------------------------------------------------------------------------
# prefill selection -> hand-off -> decode
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class HandoffReport:
    units: int = 0
    len_ok: bool = True
    rows_ok: bool = True
    budgets_ok: bool = True
    max_mu_err: float = 0.0
    max_C_err: float = 0.0
    n_err: int = 0
    min_kept: int = 0
    max_kept: int = 0
    decode: ParityReport = dataclasses.field(default_factory=ParityReport)

    def ok(self):
        return (self.len_ok and self.rows_ok and self.budgets_ok and self.n_err == 0
                and self.max_mu_err <= MOM_TOL and self.max_C_err <= MOM_TOL
                and self.decode.ok())


def run_pipeline_parity(pc: W.PrefillConfig, *, scorer: str = "snapkv", rule: int = W.RULE_EMA,
                        T: int = 1, alpha: float = 0.9, correction: int = W.CORR_FIRST_ORDER,
                        steps: int = 8, seed: int = 0, device="cuda") -> HandoffReport:
    """A prompt selected on the GPU (MomentKV's SnapKV protocol, or LaProx's
    global top-K) and handed over to a decode stream with one budget per
    (layer, KV head): the cache (kept rows in ascending position, lengths,
    budgets) and the moments of the dropped tokens against the oracle, then
    ``steps`` decode steps compared like run_decode_parity, the oracle
    evicting each unit down to its own budget."""
    from kv_cache_eviction_kvc_gb300 import kvc as K
    NL, Hq, Hkv, d, N, w, B = pc.NL, pc.Hq, pc.Hkv, pc.d, pc.N, pc.w, pc.B_total
    U, G = NL * Hkv, Hq // Hkv
    inp = W.gen_prefill_scorer(pc, device, seed)
    keep = torch.empty(NL, Hkv, N, dtype=torch.uint8, device=device)
    ws = torch.empty(K.kvc_prefill_workspace_size(NL, Hkv, N, B), dtype=torch.uint8, device=device)
    if scorer == "snapkv":
        K.kvc_prefill_snapkv(NL, Hq, Hkv, d, N, w, B, 4, 1, inp["q_win"], inp["K"], None, keep,
                             None, None, ws)
    else:
        R = torch.empty(NL, Hkv, d, d, dtype=torch.float32, device=device)
        K.kvc_prefill_prepare(NL, Hq, Hkv, d, pc.D, inp["W_O"], R)
        K.kvc_prefill_score(NL, Hq, Hkv, d, N, w, B, 1, inp["q_win"], inp["K"], inp["V"], R,
                            None, keep, None, None, ws)
    torch.cuda.synchronize()
    kh = keep.view(U, N).cpu().numpy().astype(bool)
    cnt = kh.sum(axis=1)
    budgets = np.maximum(cnt, 1).astype(np.int32)
    Lmax = int(budgets.max())
    st = DecodeState(U, G, Lmax + 2, Lmax, rule=rule, alpha=alpha, refresh_period=T,
                     correction=correction, kmax=1, device=device, budgets=True)
    ds = st.load_handoff(N, keep.view(U, N), inp["K"].view(U, N, d), inp["V"].view(U, N, d))
    torch.cuda.synchronize()
    assert ds == 0, f"hand-off device status {ds}"
    rep = HandoffReport(units=U, min_kept=int(cnt.min()), max_kept=int(cnt.max()))
    rep.budgets_ok = bool(np.array_equal(st.budget.cpu().numpy(), budgets))
    rep.len_ok = bool(np.array_equal(st.len.cpu().numpy(), cnt))
    Kb = inp["K"].view(U, N, d).cpu().view(torch.int16).numpy()
    Vb = inp["V"].view(U, N, d).cpu().view(torch.int16).numpy()
    pos_g = st.pos.cpu().numpy()
    Kg = st.K.cpu().view(torch.int16).numpy()
    Vg = st.V.cpu().view(torch.int16).numpy()
    for u in range(U):
        kept = np.nonzero(kh[u])[0]
        c = len(kept)
        if not (np.array_equal(pos_g[u, :c], kept) and np.array_equal(Kg[u, :c], Kb[u, kept])
                and np.array_equal(Vg[u, :c], Vb[u, kept])):
            rep.rows_ok = False
    # the oracle: every prompt token present, the dropped ones evicted (folded)
    sess = O.DecodeSession(U, G, d, N + steps + 2)
    try:
        for u in range(U):
            sess.load(u, Kb[u].view(np.uint16), Vb[u].view(np.uint16))
        drop = [np.nonzero(~kh[u])[0].astype(np.int32) for u in range(U)]
        kd = max(1, max(len(x) for x in drop))
        vic = np.full((U, kd), -1, np.int32)
        for u in range(U):
            vic[u, : len(drop[u])] = drop[u]
        sess.evict(vic, np.array([len(x) for x in drop], np.int32))
        n_r, mk_r, mv_r, C_r = sess.moments()
        rep.n_err += int((st.n.cpu().numpy() != n_r).sum())
        mk_g, mv_g, C_g = st.mu_k.cpu().numpy(), st.mu_v.cpu().numpy(), st.C.cpu().numpy()
        for u in range(U):
            rep.max_mu_err = max(rep.max_mu_err, _rel(mk_g[u], mk_r[u]), _rel(mv_g[u], mv_r[u]))
            rep.max_C_err = max(rep.max_C_err, _rel(C_g[u], C_r[u]))
        dc = W.DecodeConfig(f"{pc.name}-handoff", B=1, NL=NL, Hq=Hq, Hkv=Hkv, d=d, N=N, L=Lmax,
                            steps=steps, rule=rule, alpha=alpha, T=T, correction=correction)
        units = list(range(U))
        uidx = torch.arange(U, device=device)
        P = W.unit_params(dc, device, seed)
        # a unit that kept nothing starts one slot short of its budget: the
        # first step then takes the general path (max_len = Lmax + 2)
        n0 = Lmax + (1 if cnt.min() == 0 else 0)
        _step_loop(dc, st, sess, units, uidx, P, seed, device, True, steps, n0, budgets,
                   rep.decode)
    finally:
        sess.close()
    return rep
