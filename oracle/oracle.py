"""fp64 CPU oracle for the budgeted-KV decode step and the LaProx prefill scorer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its binding) never imports it
and it never imports the product path: the two share nothing but the seeded
input generators.

The arithmetic lives in ``kvc_oracle.c`` (plain C, double precision, every
function citing the passage it restates); this module compiles it with gcc,
loads it with ctypes and offers numpy-level wrappers.  A Python-level step
driver (:func:`decode_generation`) strings the C functions together in the
order of MomentKV Algorithm 1 and the InertiaKV decode loop.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, identities the pages state, brute force and library
routines (numpy).  Nothing is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvc_oracle.so")
_lock = threading.Lock()
_lib = None

RULE_SINGLE, RULE_CUMULATIVE, RULE_EMA = 0, 1, 2
RULE_MI = 3   # MomentKV moment-informed score alpha_i ||r_i||, re-scored every step
RULE_CHAINED = 4   # InertiaKV's layer-chained EMA (one state per sequence, updated per layer)
CORR_OFF, CORR_ZERO_ORDER, CORR_FIRST_ORDER = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over units).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add contraction, so the oracle
    # rounds the same way on every host architecture.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        I64 = ctypes.c_int64
        sig = {
            "ocl_create": (P, [I, I, I, I]),
            "ocl_destroy": (None, [P]),
            "ocl_load": (I, [P, I, I, P, P, P, P]),
            "ocl_append": (I, [P, P, P, ctypes.c_int32]),
            "ocl_attend": (None, [P, P, P, P, P]),
            "ocl_update_util": (None, [P, P, I, D]),
            "ocl_update_util_chained": (I, [P, P, I, I, D]),
            "ocl_get_slots": (None, [P, P, P, P, P, P]),
            "ocl_select": (I, [P, I, I, P, P, P, P]),
            "ocl_evict": (I, [P, P, P, I]),
            "ocl_zip_merge": (I, [P, P, P, ctypes.c_int32, I, D, P, P, P, P, P, P, P, P]),
            "ocl_set_row": (I, [P, I, ctypes.c_int32, P, P]),
            "ocl_get_rows": (None, [P, P, P]),
            "ocl_moments": (None, [P, P, P, P, P]),
            "ocl_mi_scores": (None, [P, P, P]),
            "ocl_mi_greedy": (I, [P, P, I, I, P, P, P, P, P, P, P]),
            "ocl_set_util": (I, [P, I, I, P]),
            "ocl_prefill_ema_init": (None, [I, I, I, I, I, I, D, P, P, P]),
            "ocl_prefill_window_colsum": (None, [I, I, I, I, I, I, P, P, P, P]),
            "ocl_snapkv_scores": (None, [I, I, I, I, I, P, P]),
            "ocl_output": (None, [P, P, I, P, P, P]),
            "ocl_prefill_gram": (None, [I, I, I, I, I, P, P]),
            "ocl_prefill_colnorm": (None, [I, I, I, I, I, I, P, P, P]),
            "ocl_prefill_rownorm": (None, [I, I, I, I, P, P, P]),
            "ocl_prefill_rownorm_direct": (None, [I, I, I, I, I, I, I, P, P, I, P, P]),
            "ocl_prefill_select": (I, [I, I, I, P, P, I, I, I64, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 array of bit patterns.

    Accepts a torch bf16 tensor (any device), a numpy uint16 array of bit
    patterns, or a float array whose values are exactly representable in bf16.
    """
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16, a.dtype
            return a.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def bf16_round(x) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); returns float64.

    Test helper for building exactly representable inputs on the CPU.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


class DecodeSession:
    """U independent (sequence, layer, KV head) units on the CPU oracle."""

    def __init__(self, U: int, G: int, d: int, cap: int):
        self.lib = _load()
        self.U, self.G, self.d, self.cap = U, G, d, cap
        self.h = self.lib.ocl_create(U, G, d, cap)
        if not self.h:
            raise MemoryError("oracle session allocation failed")

    def close(self):
        if self.h:
            self.lib.ocl_destroy(self.h)
            self.h = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def load(self, u: int, k, v, vote=None, pos=None):
        """Prefill cache of unit u: k, v [n][d] bf16; vote, pos [n] int32."""
        kb, vb = _bits(k), _bits(v)
        n = kb.shape[0]
        pos = np.arange(n, dtype=np.int32) if pos is None else np.ascontiguousarray(pos, dtype=np.int32)
        vote = None if vote is None else np.ascontiguousarray(vote, dtype=np.int32)
        rc = self.lib.ocl_load(self.h, u, n, _p(kb), _p(vb), _p(vote), _p(pos))
        if rc != 0:
            raise ValueError("ocl_load failed")

    def append(self, knew, vnew, new_pos: int):
        kb, vb = _bits(knew), _bits(vnew)
        if self.lib.ocl_append(self.h, _p(kb), _p(vb), int(new_pos)) != 0:
            raise ValueError("unit full")

    def attend(self, q):
        """Returns (lse [U][G], f [U][G][d], probs [U][cap])."""
        qb = _bits(q)
        lse = np.zeros((self.U, self.G))
        f = np.zeros((self.U, self.G, self.d))
        probs = np.zeros((self.U, self.cap))
        self.lib.ocl_attend(self.h, _p(qb), _p(lse), _p(f), _p(probs))
        return lse, f, probs

    def update_util(self, probs, rule: int, alpha: float):
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        self.lib.ocl_update_util(self.h, _p(probs), int(rule), float(alpha))

    def update_util_chained(self, probs, NL: int, Hkv: int, alpha: float):
        """InertiaKV's layer-chained EMA over each sequence's NL x Hkv units
        (see ocl_update_util_chained)."""
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        if self.lib.ocl_update_util_chained(self.h, _p(probs), int(NL), int(Hkv), float(alpha)) != 0:
            raise ValueError("chained EMA: units not grouped by sequence or lengths differ")

    def slots(self):
        """Returns (n [U], pos, vote, util, scored), each [U][cap]."""
        n = np.zeros(self.U, np.int32)
        pos = np.zeros((self.U, self.cap), np.int32)
        vote = np.zeros((self.U, self.cap), np.int32)
        util = np.zeros((self.U, self.cap))
        scored = np.zeros((self.U, self.cap), np.uint8)
        self.lib.ocl_get_slots(self.h, _p(n), _p(pos), _p(vote), _p(util), _p(scored))
        return n, pos, vote, util, scored

    def select(self, L, kmax: int):
        """Oracle's victims: (positions [U][kmax], count [U], threshold [U]).
        L: one budget, or one per unit ([U])."""
        vic = np.full((self.U, max(kmax, 1)), -1, np.int32)
        nv = np.zeros(self.U, np.int32)
        thr = np.zeros(self.U)
        Lu = None if np.isscalar(L) else np.ascontiguousarray(L, dtype=np.int32)
        rc = self.lib.ocl_select(self.h, int(L) if Lu is None else 0, max(kmax, 1), _p(vic),
                                 _p(nv), _p(thr), _p(Lu))
        if rc != 0:
            raise ValueError("ocl_select: not enough scored slots or kmax too small")
        return vic, nv, thr

    def evict(self, victims, nvict):
        victims = np.ascontiguousarray(victims, dtype=np.int32)
        nvict = np.ascontiguousarray(nvict, dtype=np.int32)
        if self.lib.ocl_evict(self.h, _p(victims), _p(nvict), victims.shape[1]) != 0:
            raise ValueError("ocl_evict: position not present")

    def zip_merge(self, q, victim, new_pos: int, R: int, eps: float = None, force=None):
        """KeepKV ZIP-merging of victim[u] (a position, -1 = none) into its
        most similar slot (see ocl_zip_merge).  Returns a dict of partner
        positions [U] (-1 = none), cos_best, cos_used [U], the unrounded
        k_r, v_r [U][d], the guard flags [U] and the weighted mean logit xt
        [U] the guard tests."""
        qb = _bits(q)
        eps = ZIP_EPS if eps is None else eps
        victim = np.ascontiguousarray(victim, dtype=np.int32)
        force = None if force is None else np.ascontiguousarray(force, dtype=np.int32)
        out = dict(partner=np.full(self.U, -1, np.int32), cos_best=np.zeros(self.U),
                   cos_used=np.zeros(self.U), kr=np.zeros((self.U, self.d)),
                   vr=np.zeros((self.U, self.d)), guard=np.zeros(self.U, np.int32),
                   xt=np.zeros(self.U))
        rc = self.lib.ocl_zip_merge(self.h, _p(qb), _p(victim), int(new_pos), int(R), float(eps),
                                    _p(force), _p(out["partner"]), _p(out["cos_best"]),
                                    _p(out["cos_used"]), _p(out["kr"]), _p(out["vr"]),
                                    _p(out["guard"]), _p(out["xt"]))
        if rc != 0:
            raise ValueError("ocl_zip_merge: victim or forced partner not present")
        return out

    def set_row(self, u: int, pos: int, k, v):
        kb, vb = _bits(k), _bits(v)
        if self.lib.ocl_set_row(self.h, int(u), int(pos), _p(kb), _p(vb)) != 0:
            raise ValueError("ocl_set_row: position not present")

    def rows(self):
        """Key and value rows [U][cap][d] as bf16 bit patterns (slot order)."""
        k = np.zeros((self.U, self.cap, self.d), np.uint16)
        v = np.zeros((self.U, self.cap, self.d), np.uint16)
        self.lib.ocl_get_rows(self.h, _p(k), _p(v))
        return k, v

    def set_util(self, u: int, util):
        """Utilities of unit u's first len(util) slots (marked scored)."""
        util = np.ascontiguousarray(util, dtype=np.float64)
        if self.lib.ocl_set_util(self.h, int(u), int(util.shape[0]), _p(util)) != 0:
            raise ValueError("ocl_set_util: more utilities than slots")

    def mi_scores(self, probs):
        """MomentKV moment-informed scores alpha_i ||r_i|| [U][cap] from the
        attention weights probs [U][cap] and the session's moments."""
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        out = np.zeros((self.U, self.cap))
        self.lib.ocl_mi_scores(self.h, _p(probs), _p(out))
        return out

    def mi_greedy(self, q, L, kmax: int, forced=None):
        """MomentKV Algorithm 1 phase 1 on every unit: while a unit holds more
        than L slots, score every slot (alpha ||r|| with alpha re-formed over
        the slots present and the moments as they stand), evict the lowest
        and fold it (see ocl_mi_greedy).  ``forced`` [U][kmax] (positions in
        eviction order) replays another implementation's choices.  Returns a
        dict: victims [U][kmax] (eviction order), nvict [U], best / used
        [U][kmax] (each round's lowest score and the removed slot's score),
        scores0 [U][cap] (first-round scores, slot order before the step)."""
        qb = _bits(q)
        kmax = max(1, int(kmax))
        forced = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        if forced is not None and forced.shape != (self.U, kmax):
            raise ValueError("forced must be [U][kmax]")
        out = dict(victims=np.full((self.U, kmax), -1, np.int32),
                   nvict=np.zeros(self.U, np.int32), best=np.zeros((self.U, kmax)),
                   used=np.zeros((self.U, kmax)), scores0=np.zeros((self.U, self.cap)))
        Lu = None if np.isscalar(L) else np.ascontiguousarray(L, dtype=np.int32)
        rc = self.lib.ocl_mi_greedy(self.h, _p(qb), int(L) if Lu is None else 0, kmax,
                                    _p(forced), _p(out["victims"]), _p(out["nvict"]),
                                    _p(out["best"]), _p(out["used"]), _p(out["scores0"]),
                                    _p(Lu))
        if rc != 0:
            raise ValueError("ocl_mi_greedy: kmax too small or a forced position is not present")
        return out

    def moments(self):
        """Returns (n [U], mu_k [U][d], mu_v [U][d], C [U][d][d])."""
        n = np.zeros(self.U)
        mk = np.zeros((self.U, self.d))
        mv = np.zeros((self.U, self.d))
        C = np.zeros((self.U, self.d, self.d))
        self.lib.ocl_moments(self.h, _p(n), _p(mk), _p(mv), _p(C))
        return n, mk, mv, C

    def output(self, q, correction: int):
        """Returns (o, f_R [U][G][d], logZ_R [U][G])."""
        qb = _bits(q)
        o = np.zeros((self.U, self.G, self.d))
        fR = np.zeros((self.U, self.G, self.d))
        lz = np.zeros((self.U, self.G))
        self.lib.ocl_output(self.h, _p(qb), int(correction), _p(o), _p(fR), _p(lz))
        return o, fR, lz


# Guard of the ZIP-merge key formula on the weighted mean logit (KeepKV
# reading notes, "numerical stability" item 2; the pages give no value).
ZIP_EPS = 1e-3


def is_refresh(t: int, T: int) -> bool:
    """Refresh steps: t = 1 and every T-th step after it (t - 1 = 0 mod T)
    [InertiaKV abstract / sec 1, InertiaKV-Lazy periodic refresh; reading:
    utilities are refreshed on those steps only and are stale in between].
    T = 0 is Score-Free (InertiaKV abstract and sec 1): scored at the first
    decode step, then frozen."""
    if T == 0:
        return t == 1
    return T == 1 or (t - 1) % T == 0


def decode_step(sess: DecodeSession, t: int, new_pos: int, q, knew, vnew, *,
                L, rule: int, alpha: float, T: int, correction: int,
                choose=None, merge_recent: int | None = None, force_partner=None,
                mi_forced=None, chain=None):
    """One decode step on every unit of ``sess``, in the order of MomentKV
    Algorithm 1 with the InertiaKV utility in place of its scoring:

    1. append (k_new, v_new) with vote 1
    2. vote-weighted attention over all slots -> lse, f_all, head-mean probs
    3. refresh step: utility update                 (InertiaKV sec 3.1 eqs 2-4)
    4. victims: the k = n - L lowest (utility, position) scored slots
    5. fold victims into the moments and remove them  (eviction phase)
    6. retained attention + moment correction         (inference phase)

    Under rule RULE_MI steps 3-5 are MomentKV's moment-aware eviction phase
    itself (Algorithm 1 phase 1, :meth:`DecodeSession.mi_greedy`): every
    step, while a unit holds more than L slots, score alpha ||r|| over the
    slots present, evict the lowest, fold it, and score again.
    ``mi_forced`` [U][kmax] (positions in eviction order) replays another
    implementation's choices; the result's ``mi_best`` / ``mi_used`` give
    each round's lowest score and the score of the slot removed.

    ``L`` is one budget or one per unit ([U]; a cache handed over from a
    prefill scorer keeps each unit at its own length).

    Under rule RULE_CHAINED (InertiaKV's layer-chained EMA) ``chain`` =
    (NL, Hkv) groups the units by sequence; one utility per slot of a
    sequence, so every unit of it evicts the same slots.

    ``choose(t, proposal)``, if given, receives the oracle's proposal dict and
    returns the victim positions to apply ([U][kmax], [U]); tests use it to
    validate a near-tie alternative before adopting it (not under RULE_MI).

    ``merge_recent = R`` (not None) selects KeepKV ZIP-merging: a unit that
    removes exactly one slot this step merges its victim into the most
    similar slot outside the last R positions instead of dropping it (no
    moment fold), and its output is the one over the cache before the merge
    (KeepKV Algorithm 1, decoding stage: attend, then compress; by KeepKV
    Thm 3 the merged cache gives the same output for the group's mean
    query).  Units that remove more than one slot, or find no partner, evict
    as above.  ``force_partner`` [U] (positions, -1 = the oracle's own
    choice) makes the oracle merge into a given slot; the result's
    ``merge["cos_best"]`` and ``merge["cos_used"]`` let the caller check that
    the forced choice is within a near-tie of the best.
    """
    sess.append(knew, vnew, new_pos)
    lse, f_all, probs = sess.attend(q)
    if rule == RULE_MI:
        if merge_recent is not None:
            raise ValueError("the moment-informed rule evicts; it is not combined with merging")
        n = sess.slots()[0]
        kmax = int(max(1, (n - np.asarray(L)).max()))
        if mi_forced is not None:
            mi_forced = np.asarray(mi_forced)
            kmax = max(kmax, mi_forced.shape[1])
            f = np.full((sess.U, kmax), -1, np.int32)
            f[:, : mi_forced.shape[1]] = mi_forced
            mi_forced = f
        g = sess.mi_greedy(q, L, kmax, forced=mi_forced)
        vic, nv = g["victims"], g["nvict"]
        last = np.maximum(nv - 1, 0)
        thr = np.where(nv > 0, g["best"][np.arange(sess.U), last], 0.0)
        proposal = dict(victims=vic, nvict=nv, thr=thr, lse=lse, f_all=f_all, probs=probs,
                        refresh=True, mi_scores=g["scores0"], mi_best=g["best"],
                        mi_used=g["used"])
    else:
        refresh = is_refresh(t, T)
        if refresh and rule == RULE_CHAINED:
            sess.update_util_chained(probs, chain[0], chain[1], alpha)
        elif refresh:
            sess.update_util(probs, rule, alpha)
        n = sess.slots()[0]
        kmax = int(max(1, (n - np.asarray(L)).max()))
        vic, nv, thr = sess.select(L, kmax)
        proposal = dict(victims=vic, nvict=nv, thr=thr, lse=lse, f_all=f_all,
                        probs=probs if refresh else None, refresh=refresh, mi_scores=None)
        if choose is not None:
            vic, nv = choose(t, proposal)
    merged = np.zeros(len(nv), bool)
    if merge_recent is not None:
        o0, fR0, lz0 = sess.output(q, correction)       # every slot, before the merge
        victim = np.where(np.asarray(nv) == 1, np.asarray(vic)[:, 0], -1)
        mres = sess.zip_merge(q, victim, new_pos, merge_recent, force=force_partner)
        merged = mres["partner"] >= 0
        proposal.update(merge=mres, merged=merged)
        nv = np.where(merged, 0, nv).astype(np.int32)
    if rule != RULE_MI:                 # the moment-aware phase already evicted
        sess.evict(vic, nv)
    o, fR, lz = sess.output(q, correction)
    if merge_recent is not None:
        o[merged], fR[merged], lz[merged] = o0[merged], fR0[merged], lz0[merged]
    proposal.update(o=o, f_R=fR, logZ_R=lz, applied_victims=vic, applied_nvict=nv,
                    merged=merged)
    return proposal


def decode_generation(k_pre, v_pre, q_steps, k_steps, v_steps, *, L: int,
                      rule: int, alpha: float, T: int, correction: int,
                      votes_pre=None, G: int | None = None, cap: int | None = None,
                      merge_recent: int | None = None):
    """Run a whole generation on the oracle with its own decisions.

    k_pre, v_pre: [U][N][d]; q_steps: [S][U][G][d]; k_steps, v_steps: [S][U][d]
    (bf16 bit patterns or bf16-exact floats).  Returns a list of per-step
    result dicts (see :func:`decode_step`).
    """
    kp, vp = _bits(k_pre), _bits(v_pre)
    U, N, d = kp.shape
    qs = _bits(q_steps)
    S = qs.shape[0]
    G = qs.shape[2] if G is None else G
    cap = (N + S) if cap is None else cap
    sess = DecodeSession(U, G, d, cap)
    try:
        for u in range(U):
            vote = None if votes_pre is None else np.asarray(votes_pre[u])
            sess.load(u, kp[u], vp[u], vote)
        ks, vs = _bits(k_steps), _bits(v_steps)
        out = []
        for s in range(S):
            t = s + 1
            out.append(decode_step(sess, t, N + t - 1, qs[s], ks[s], vs[s], L=L,
                                   rule=rule, alpha=alpha, T=T,
                                   correction=correction, merge_recent=merge_recent))
            out[-1]["moments"] = sess.moments()
        return out
    finally:
        sess.close()


# ---------------------------------------------------------------------------
# prefill scorer
# ---------------------------------------------------------------------------

def prefill_gram(W_O, NL: int, Hq: int, Hkv: int, d: int) -> np.ndarray:
    wb = _bits(W_O)
    D = wb.shape[-1]
    out = np.zeros((NL, Hkv, d, d))
    _load().ocl_prefill_gram(NL, Hq, Hkv, d, D, _p(wb), _p(out))
    return out


def prefill_colnorm(q_win, K, NL: int, Hq: int, Hkv: int, d: int, N: int, w: int):
    qb, kb = _bits(q_win), _bits(K)
    out = np.zeros((NL, Hkv, N))
    _load().ocl_prefill_colnorm(NL, Hq, Hkv, d, N, w, _p(qb), _p(kb), _p(out))
    return out


def prefill_rownorm(V, Gram, NL: int, Hkv: int, d: int, N: int):
    vb = _bits(V)
    Gram = np.ascontiguousarray(Gram, dtype=np.float64)
    out = np.zeros((NL, Hkv, N))
    _load().ocl_prefill_rownorm(NL, Hkv, d, N, _p(vb), _p(Gram), _p(out))
    return out


def prefill_rownorm_direct(V, W_O, Hq: int, Hkv: int, d: int, N: int, l: int,
                           g: int, tokens):
    vb, wb = _bits(V), _bits(W_O)
    D = wb.shape[-1]
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.zeros(tokens.shape[0])
    _load().ocl_prefill_rownorm_direct(Hq, Hkv, d, D, N, l, g, _p(vb), _p(wb),
                                       tokens.shape[0], _p(tokens), _p(out))
    return out


# budget allocations of the LaProx ablation: global (head- and layer-flatten),
# per layer (head-flatten only), uniform per head
ALLOC_GLOBAL, ALLOC_LAYER, ALLOC_HEAD = 0, 1, 2


def prefill_select(c, r, B_total: int, normalize: bool = True, alloc: int = ALLOC_GLOBAL):
    """Selection of the LaProx scorer; ``thr`` is a float for the global
    allocation and an array (one threshold per segment) otherwise."""
    c = np.ascontiguousarray(c, dtype=np.float64)
    r = np.ascontiguousarray(r, dtype=np.float64)
    NL, Hkv, N = c.shape
    s = np.zeros_like(c)
    keep = np.zeros(c.shape, np.uint8)
    counts = np.zeros((NL, Hkv), np.int32)
    idx = np.zeros(max(int(B_total), 1), np.int64)
    nseg = 1 if alloc == ALLOC_GLOBAL else NL if alloc == ALLOC_LAYER else NL * Hkv
    thr = np.zeros(nseg)
    rc = _load().ocl_prefill_select(NL, Hkv, N, _p(c), _p(r), int(bool(normalize)), int(alloc),
                                    int(B_total), _p(s), _p(keep), _p(counts),
                                    _p(idx), _p(thr))
    if rc != 0:
        raise ValueError("B_total out of range or not a multiple of the segments")
    return dict(s=s, keep=keep, counts=counts, idx=idx[:int(B_total)],
                thr=float(thr[0]) if alloc == ALLOC_GLOBAL else thr)


def prefill_ema_init(q_win, K, NL: int, Hq: int, Hkv: int, d: int, N: int, w: int,
                     alpha: float) -> np.ndarray:
    """KeepKV windowed EMA initialization of the utilities, S [NL][Hkv][N]
    (see ocl_prefill_ema_init)."""
    qb, kb = _bits(q_win), _bits(K)
    S = np.zeros((NL, Hkv, N))
    _load().ocl_prefill_ema_init(NL, Hq, Hkv, d, N, w, float(alpha), _p(qb), _p(kb), _p(S))
    return S


def prefill_window_colsum(q_win, K, NL: int, Hq: int, Hkv: int, d: int, N: int, w: int,
                          roww) -> np.ndarray:
    """Weighted column sum of the group-mean window attention,
    S [NL][Hkv][N] (see ocl_prefill_window_colsum)."""
    qb, kb = _bits(q_win), _bits(K)
    roww = np.ascontiguousarray(roww, dtype=np.float64)
    assert roww.shape == (w,)
    S = np.zeros((NL, Hkv, N))
    _load().ocl_prefill_window_colsum(NL, Hq, Hkv, d, N, w, _p(roww), _p(qb), _p(kb), _p(S))
    return S


def snapkv_scores(acc, pool: int = 4, sink: bool = True) -> np.ndarray:
    """SnapKV scores under MomentKV's prefill protocol: block means of the
    accumulated window attention, sink at position 0 (see ocl_snapkv_scores)."""
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    NL, Hkv, N = acc.shape
    s = np.zeros_like(acc)
    _load().ocl_snapkv_scores(NL, Hkv, N, int(pool), int(bool(sink)), _p(acc), _p(s))
    return s


def prefill_snapkv(q_win, K, *, NL: int, Hq: int, Hkv: int, d: int, N: int, w: int,
                   B_total: int, pool: int = 4, sink: bool = True):
    """MomentKV's SnapKV prefill protocol: attention accumulated over the
    observation window, block pooling, the sink kept, and each layer's
    budget B_total / NL shared by its heads (adaptive per-head allocation
    within the layer)."""
    acc = prefill_window_colsum(q_win, K, NL, Hq, Hkv, d, N, w, np.ones(w))
    sc = snapkv_scores(acc, pool, sink)
    res = prefill_select(sc, np.ones_like(sc), B_total, normalize=False, alloc=ALLOC_LAYER)
    res.update(acc=acc, scores=sc)
    return res


def prefill_score(q_win, K, V, W_O, *, NL: int, Hq: int, Hkv: int, d: int,
                  N: int, w: int, B_total: int, normalize: bool = True,
                  alloc: int = ALLOC_GLOBAL):
    """Whole LaProx prefill scorer on the oracle (Gram route for r)."""
    Gram = prefill_gram(W_O, NL, Hq, Hkv, d)
    c = prefill_colnorm(q_win, K, NL, Hq, Hkv, d, N, w)
    r = prefill_rownorm(V, Gram, NL, Hkv, d, N)
    res = prefill_select(c, r, B_total, normalize, alloc)
    res.update(c=c, r=r, Gram=Gram)
    return res
