"""Device-memory plumbing for a decode stream: allocates the cache, moment,
workspace and output tensors with torch and calls the libkvc entry points
through the binding.  No arithmetic of the method happens here."""
from __future__ import annotations

import torch

from . import kvc as K_


class DecodeState:
    """Cache + moments + workspace of U units on one device."""

    def __init__(self, U: int, G: int, cap: int, L: int, *, rule: int = K_.RULE_EMA,
                 alpha: float = 0.9, refresh_period: int = 1,
                 correction: int = K_.CORR_FIRST_ORDER, votes: bool = False,
                 kmax: int = 1, device="cuda", d: int = 128, merge_recent: int | None = None,
                 budgets: bool = False, chain=None):
        self.U, self.G, self.cap, self.L, self.d = U, G, cap, L, d
        self.device = torch.device(device)
        # per-unit budgets (a cache handed over from a prefill selection);
        # the tensor lives as long as the parameters that point at it
        self.budget = (torch.full((U,), L, dtype=torch.int32, device=self.device)
                       if budgets else None)
        self.params = K_.make_params(U, G, cap, L, rule, alpha, refresh_period, correction, d,
                                     merge_recent, self.budget, chain)
        self.merge = merge_recent is not None
        if self.merge and not votes:
            raise ValueError("ZIP-merging needs per-slot votes (votes=True)")
        dev = self.device
        self.K = torch.zeros(U, cap, d, dtype=torch.bfloat16, device=dev)
        self.V = torch.zeros(U, cap, d, dtype=torch.bfloat16, device=dev)
        self.votes = torch.ones(U, cap, dtype=torch.int32, device=dev) if votes else None
        self.pos = torch.full((U, cap), -1, dtype=torch.int32, device=dev)
        self.util = torch.full((U, cap), float("inf"), dtype=torch.float64, device=dev)
        self.len = torch.zeros(U, dtype=torch.int32, device=dev)
        self.n = torch.zeros(U, dtype=torch.float32, device=dev)
        self.mu_k = torch.zeros(U, d, dtype=torch.float32, device=dev)
        self.mu_v = torch.zeros(U, d, dtype=torch.float32, device=dev)
        self.C = torch.zeros(U, d, d, dtype=torch.float32, device=dev)
        nbytes = K_.kvc_decode_workspace_size(self.params)
        if nbytes == 0:
            raise K_.KvcError(1, "invalid decode parameters")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        K_.kvc_decode_workspace_init(self.params, self.ws)
        self.o = torch.zeros(U, G, d, dtype=torch.float32, device=dev)
        self.probs = torch.zeros(U, cap, dtype=torch.float64, device=dev)
        self.lse = torch.zeros(U, G, dtype=torch.float32, device=dev)
        self.f_all = torch.zeros(U, G, d, dtype=torch.float32, device=dev)
        self.f_R = torch.zeros(U, G, d, dtype=torch.float32, device=dev)
        self.logZ_R = torch.zeros(U, G, dtype=torch.float32, device=dev)
        self.n_evict = torch.zeros(U, dtype=torch.int32, device=dev)
        self.partner_pos = torch.full((U,), -1, dtype=torch.int32, device=dev)
        self.scores = (torch.zeros(U, cap, dtype=torch.float64, device=dev)
                       if rule == K_.RULE_MI else None)
        self.set_kmax(kmax)

    # --------------------------------------------------------------- helpers
    def set_kmax(self, kmax: int):
        kmax = max(1, int(kmax))
        if getattr(self, "kmax", 0) != kmax:
            self.kmax = kmax
            self.evict_idx = torch.full((self.U, kmax), -1, dtype=torch.int32, device=self.device)
            self.evict_pos = torch.full((self.U, kmax), -1, dtype=torch.int32, device=self.device)

    @property
    def cache(self) -> K_.kvc_cache:
        return K_.make_cache(self.K, self.V, self.votes, self.pos, self.util, self.len)

    @property
    def moments(self) -> K_.kvc_moments:
        return K_.make_moments(self.n, self.mu_k, self.mu_v, self.C)

    def load_prefill(self, K, V, votes, pos, length):
        """Copy a prefill cache laid out [U][>=N][d] into the state."""
        n = K.shape[1]
        if K.data_ptr() != self.K.data_ptr():      # drawn in place: nothing to copy
            self.K[:, :n].copy_(K)
        if V.data_ptr() != self.V.data_ptr():
            self.V[:, :n].copy_(V)
        if self.votes is not None and votes is not None:
            self.votes[:, :n].copy_(votes[:, :n])
        self.pos[:, :n].copy_(pos[:, :n])
        self.util.fill_(float("inf"))
        self.len.copy_(length)
        for t in (self.n, self.mu_k, self.mu_v, self.C):
            t.zero_()

    def load_handoff(self, N, keep, K_src, V_src, votes_src=None, util_init=None):
        """Start the stream from a prefill selection (kvc_prefill_handoff):
        keep [U][N] uint8, K_src / V_src [U][N][d]; the per-unit budgets land
        in self.budget.  Returns the device status of the call."""
        ws = torch.empty(K_.kvc_prefill_handoff_workspace_size(self.U, N), dtype=torch.uint8,
                         device=self.device)
        K_.kvc_prefill_handoff(self.params, N, keep, K_src, V_src, votes_src, util_init,
                               self.cache, self.moments, self.budget, ws)
        return K_.kvc_get_device_status(ws)

    def device_status(self) -> int:
        return K_.kvc_get_device_status(self.ws)

    # --------------------------------------------------------------- steps
    def step(self, t: int, new_pos: int, q, k_new, v_new, max_len: int, emit_probs=True,
             stream=None, o=None):
        """Fused kvc_decode_step (falls back to the five-call sequence inside
        the library when the step is not in the steady state).  `o` may name
        another [U][G][d] fp32 output buffer."""
        self.set_kmax(max_len - self.L)
        K_.kvc_decode_step(self.params, t, new_pos, max_len, q, k_new, v_new, self.cache,
                           self.moments, self.o if o is None else o,
                           self.probs if emit_probs else None,
                           self.kmax, self.evict_idx, self.evict_pos, self.n_evict, self.ws,
                           stream)

    def step_calls(self, t: int, new_pos: int, q, k_new, v_new, max_len: int, stream=None):
        """The five entry points in order (attend, aggregate_evict,
        moment_update, correct, compact), with zip_merge after aggregate_evict
        in merge mode and mi_scores before it under the moment-informed rule
        (mi_evict in place of scores, aggregate and fold when that rule
        removes several slots)."""
        self.set_kmax(max_len - self.L)
        c = self.cache
        K_.kvc_decode_attend(self.params, t, new_pos, max_len, q, k_new, v_new, c, self.lse,
                             self.f_all, self.probs, self.ws, stream)
        mi = self.params.rule == K_.RULE_MI          # the rule of this step
        if mi and max_len - self.L > 1:
            # MomentKV Algorithm 1's loop: score, evict the lowest, fold, again
            K_.kvc_mi_evict(self.params, max_len, c, self.moments, self.lse, self.kmax,
                            self.evict_idx, self.evict_pos, self.n_evict, self.ws, stream)
            K_.kvc_correct(self.params, q, c, self.kmax, self.evict_idx, self.n_evict, self.lse,
                           self.f_all, self.moments, self.o, self.f_R, self.logZ_R, self.ws,
                           stream)
            K_.kvc_compact(self.params, c, self.kmax, self.evict_idx, self.n_evict, self.ws,
                           stream)
            return
        agg_in = self.probs
        if mi:
            K_.kvc_mi_scores(self.params, c, self.moments, max_len, self.probs, self.scores, stream)
            agg_in = self.scores
        K_.kvc_aggregate_evict(self.params, t, agg_in, c, self.kmax, self.evict_idx,
                               self.evict_pos, self.n_evict, self.ws, stream)
        if self.merge:
            K_.kvc_zip_merge(self.params, new_pos, q, c, self.kmax, self.evict_idx, self.n_evict,
                             self.partner_pos, self.ws, stream)
        K_.kvc_moment_update(self.params, c, self.kmax, self.evict_idx, self.n_evict,
                             self.moments, self.ws, stream)
        K_.kvc_correct(self.params, q, c, self.kmax, self.evict_idx, self.n_evict, self.lse,
                       self.f_all, self.moments, self.o, self.f_R, self.logZ_R, self.ws, stream)
        K_.kvc_compact(self.params, c, self.kmax, self.evict_idx, self.n_evict, self.ws, stream)
