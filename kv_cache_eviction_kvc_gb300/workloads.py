"""Seeded synthetic workloads for the budgeted-KV decode step and the prefill
scorer.

This module only draws random numbers; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may take their inputs
from it.  Every tensor is bf16 (votes and positions int32), generated with
``torch.Generator`` on the requested device from a fixed seed plus a fixed
per-tensor offset.

Shapes follow the attention geometry the pages evaluate: Llama-3.1-8B and
Qwen3-4B both have 32 query heads over 8 KV heads and head dimension 128
(MomentKV experimental setup, "models").  Value distributions are the ones
the decode configs name:

* ``normal``: N(0, 1).
* ``mixture``: each token draws a component index c uniformly from
  ``centres`` components; K = centre_K[c] + sigma * N(0,1), V = centre_V[c] +
  sigma * N(0,1), the index shared by K and V of the token and the centres
  N(0, 1), drawn once per unit (sequence, layer, KV head).
* ``head_scale``: a per-unit factor U(lo, hi) multiplying Q, K and V of the
  unit's query group; ``outliers`` channels per unit (drawn once from the
  seed) multiplied by ``outlier_mult`` in Q, K and V.

The real workloads of the pages (LongBench, RULER, needle-in-a-haystack on
Llama / Qwen activations) are not available here; these inputs stand in for
them by shape, size and value structure only.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

RULE_SINGLE, RULE_CUMULATIVE, RULE_EMA, RULE_MI, RULE_EMA_CHAINED = 0, 1, 2, 3, 4
CORR_OFF, CORR_ZERO_ORDER, CORR_FIRST_ORDER = 0, 1, 2

# fixed per-tensor seed offsets
_OFF_UNIT = 11      # per-unit parameters (centres, scales, outlier channels)
_OFF_PREFILL = 23   # prefill K / V / votes
_OFF_STEP = 1009    # decode-step q / k_new / v_new (plus the step index)
_OFF_PRE_Q = 31     # prefill-scorer window queries
_OFF_PRE_KV = 37    # prefill-scorer K / V
_OFF_PRE_W = 41     # prefill-scorer W_O


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    NL: int
    Hq: int
    Hkv: int
    d: int
    N: int
    L: int
    steps: int
    rule: int = RULE_EMA
    alpha: float = 0.9
    T: int = 1
    correction: int = CORR_FIRST_ORDER
    votes_max: int = 0          # 0: no votes; else p ~ U{1..votes_max} on prefill slots
    k_dist: str = "normal"
    v_dist: str = "normal"
    centres: int = 0
    sigma: float = 0.3
    head_scale: tuple | None = None
    outliers: int = 0
    outlier_mult: float = 8.0
    merge_recent: int | None = None   # KeepKV ZIP-merging, last R positions excluded
    first_rule: int | None = None     # rule of the first decode step (None: ``rule``)
    description: str = ""

    @property
    def U(self) -> int:
        return self.B * self.NL * self.Hkv

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "DecodeConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    NL: int
    Hq: int
    Hkv: int
    d: int
    N: int
    w: int
    B_total: int
    wo_std: float = 1.0 / 64.0
    description: str = ""
    D_out: int = 0            # output width of W_O; 0 = Hq * d (the model width)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def D(self) -> int:
        return self.D_out or self.Hq * self.d

    def with_(self, **kw) -> "PrefillConfig":
        return replace(self, **kw)


C0 = DecodeConfig(
    "C0-tiny", B=1, NL=1, Hq=8, Hkv=2, d=128, N=512, L=64, steps=32,
    rule=RULE_EMA, alpha=0.9, T=1, k_dist="normal", v_dist="mixture",
    centres=16, sigma=0.3,
    description="1 seq, 1 layer, 8 q / 2 KV heads, N=512, L=64, 32 steps, "
                "V 16-centre mixture, EMA 0.9")
C1 = DecodeConfig(
    "C1-llama8b", B=1, NL=32, Hq=32, Hkv=8, d=128, N=4096, L=128, steps=256,
    rule=RULE_EMA, alpha=0.9, T=1, head_scale=(0.5, 2.0), outliers=4,
    outlier_mult=8.0,
    description="Llama-3.1-8B attention shape, batch 1, N=4096, L=128, 256 "
                "steps, per-head scales U(0.5,2), 4 outlier channels x8, EMA 0.9")
C2 = DecodeConfig(
    "C2-qwen3-4b", B=16, NL=36, Hq=32, Hkv=8, d=128, N=32768, L=3277,
    steps=512, rule=RULE_EMA, alpha=0.9, T=8, k_dist="mixture",
    v_dist="mixture", centres=64, sigma=0.3,
    description="Qwen3-4B attention shape, batch 16, N=32768, L=3277 (10%), "
                "512 steps, lazy refresh every 8 steps, K/V 64-centre mixture")
C4 = DecodeConfig(
    "C4-long", B=8, NL=32, Hq=32, Hkv=8, d=128, N=131072, L=1024,
    steps=1024, rule=RULE_EMA, alpha=0.95, T=1, votes_max=8,
    k_dist="mixture", v_dist="mixture", centres=64, sigma=0.3,
    description="batch 8, 32 layers, N=131072, L=1024, 1024 steps, votes "
                "U{1..8}, K/V 64-centre mixture, EMA 0.95")
C3 = PrefillConfig(
    "C3-prefill", NL=32, Hq=32, Hkv=8, d=128, N=16384, w=32,
    B_total=128 * 32 * 8,
    description="prefill scoring: 32 layers, 32 q / 8 KV heads, N=16384, "
                "window 32, W_O 4096x4096 ~ N(0, 1/4096), global top-K 32768")

# variants of the Qwen3-4B decode workload for the aggregation and merging
# rows: Score-Free (InertiaKV: scored at the first decode step only) and
# KeepKV ZIP-merging (partners outside the last 32 positions)
C2_SCORE_FREE = C2.with_(name="C2-qwen3-4b-score-free", T=0,
                         description=C2.description.replace("lazy refresh every 8 steps",
                                                            "Score-Free (no refresh after step 1)"))
C2_ZIP = C2.with_(name="C2-qwen3-4b-zip", merge_recent=32,
                  description=C2.description + ", KeepKV ZIP-merging (R = 32)")

# MomentKV's moment-informed eviction (alpha ||r|| every step) on the same
# shape.  The 32768-token prompt is first brought to the budget by one
# attention-scored eviction at the first decode step (MomentKV's own setup
# compresses the prompt before decoding, with the SnapKV protocol); the
# moment-aware loop then removes one slot per step.
C2_MI = C2.with_(name="C2-qwen3-4b-mi", rule=RULE_MI, T=1, first_rule=RULE_EMA,
                 description=C2.description.replace(
                     "lazy refresh every 8 steps",
                     "prompt compressed by attention at step 1, then MomentKV "
                     "moment-informed eviction every step"))

# InertiaKV's layer-chained EMA on the Llama-3.1-8B shape: one utility state
# per sequence, carried from layer to layer of each step
C1_CHAINED = C1.with_(name="C1-llama8b-chained", rule=RULE_EMA_CHAINED,
                      description=C1.description.replace("EMA 0.9",
                                                         "layer-chained EMA 0.9"))

DECODE_CONFIGS = {"C0": C0, "C1": C1, "C2": C2, "C4": C4,
                  "C2-score-free": C2_SCORE_FREE, "C2-zip": C2_ZIP, "C2-mi": C2_MI,
                  "C1-chained": C1_CHAINED}
PREFILL_CONFIGS = {"C3": C3}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _chunk_units(cfg: DecodeConfig) -> int:
    # bound the fp32 intermediates of one chunk to ~512 MB; depends on the
    # config only, so the drawn numbers never depend on the device
    per_unit = max(1, (cfg.N + 1) * cfg.d * 4 * 3)
    return max(1, min(cfg.U, (512 << 20) // per_unit))


@dataclass
class UnitParams:
    """Per-unit random parameters (on the generation device)."""
    centres_k: torch.Tensor | None = None   # [U][C][d] fp32
    centres_v: torch.Tensor | None = None
    scale: torch.Tensor | None = None        # [U] fp32
    outlier_mask: torch.Tensor | None = None  # [U][d] fp32 multipliers
    extra: dict = field(default_factory=dict)


def unit_params(cfg: DecodeConfig, device, seed: int = 0) -> UnitParams:
    g = _gen(device, seed * 7919 + _OFF_UNIT)
    U, d = cfg.U, cfg.d
    p = UnitParams()
    if cfg.centres:
        p.centres_k = torch.randn(U, cfg.centres, d, generator=g, device=device)
        p.centres_v = torch.randn(U, cfg.centres, d, generator=g, device=device)
    if cfg.head_scale is not None:
        lo, hi = cfg.head_scale
        p.scale = lo + (hi - lo) * torch.rand(U, generator=g, device=device)
    if cfg.outliers:
        m = torch.ones(U, d, device=device)
        r = torch.rand(U, d, generator=g, device=device)
        idx = r.argsort(dim=1)[:, : cfg.outliers]
        m.scatter_(1, idx, cfg.outlier_mult)
        p.outlier_mask = m
    return p


def _draw_kv(cfg: DecodeConfig, P: UnitParams, u0: int, u1: int, n: int,
             g: torch.Generator, device):
    """Draw n tokens of K and V for units [u0, u1); fp32 [u][n][d]."""
    nu, d = u1 - u0, cfg.d
    comp = None
    if "mixture" in (cfg.k_dist, cfg.v_dist):
        comp = torch.randint(0, cfg.centres, (nu, n), generator=g, device=device)
    out = []
    for dist, centres in ((cfg.k_dist, P.centres_k), (cfg.v_dist, P.centres_v)):
        x = torch.randn(nu, n, d, generator=g, device=device)
        if dist == "mixture":
            c = torch.gather(centres[u0:u1], 1,
                             comp.unsqueeze(-1).expand(nu, n, d))
            x = c + cfg.sigma * x
        out.append(x)
    k, v = out
    if P.scale is not None:
        s = P.scale[u0:u1].view(nu, 1, 1)
        k, v = k * s, v * s
    if P.outlier_mask is not None:
        m = P.outlier_mask[u0:u1].view(nu, 1, d)
        k, v = k * m, v * m
    return k, v


def gen_prefill(cfg: DecodeConfig, device, seed: int = 0, cap: int | None = None,
                P: UnitParams | None = None, out_K=None, out_V=None):
    """Prefill cache of every unit.

    Returns dict with K, V [U][cap][d] bf16 (slots [0, N) filled, the rest
    zero), votes [U][cap] int32 or None (prefill slots U{1..votes_max}, the rest
    1), pos [U][cap] int32 (prefill slot i holds position i, the rest -1),
    len [U] int32 = N.  ``out_K`` / ``out_V`` (bf16 [U][cap][d]) receive the
    draw in place of new tensors (slots past N untouched), so a large cache is
    drawn straight into its final buffers; the numbers do not change.
    """
    cap = cfg.N + 1 if cap is None else cap
    assert cap >= cfg.N
    P = unit_params(cfg, device, seed) if P is None else P
    U, N, d = cfg.U, cfg.N, cfg.d
    if out_K is not None:
        assert out_K.shape == (U, cap, d) and out_V is not None and out_V.shape == out_K.shape
        K, V = out_K, out_V
    else:
        K = torch.zeros(U, cap, d, dtype=torch.bfloat16, device=device)
        V = torch.zeros(U, cap, d, dtype=torch.bfloat16, device=device)
    g = _gen(device, seed * 7919 + _OFF_PREFILL)
    cu = _chunk_units(cfg)
    for u0 in range(0, U, cu):
        u1 = min(U, u0 + cu)
        k, v = _draw_kv(cfg, P, u0, u1, N, g, device)
        K[u0:u1, :N] = k.to(torch.bfloat16)
        V[u0:u1, :N] = v.to(torch.bfloat16)
        del k, v
    votes = None
    if cfg.votes_max:
        votes = torch.ones(U, cap, dtype=torch.int32, device=device)
        votes[:, :N] = torch.randint(1, cfg.votes_max + 1, (U, N), generator=g,
                                     device=device, dtype=torch.int32)
    pos = torch.full((U, cap), -1, dtype=torch.int32, device=device)
    pos[:, :N] = torch.arange(N, dtype=torch.int32, device=device)
    length = torch.full((U,), N, dtype=torch.int32, device=device)
    return dict(K=K, V=V, votes=votes, pos=pos, len=length, params=P)


def gen_step(cfg: DecodeConfig, device, t: int, seed: int = 0,
             P: UnitParams | None = None):
    """Inputs of decode step t (1-based): q [U][G][d], k_new, v_new [U][d] bf16.

    Queries are N(0,1) (times the unit's scale and outlier channels where the
    config has them); the new key and value follow the prefill distribution.
    """
    P = unit_params(cfg, device, seed) if P is None else P
    U, G, d = cfg.U, cfg.G, cfg.d
    g = _gen(device, seed * 7919 + _OFF_STEP + 131 * t)
    q = torch.randn(U, G, d, generator=g, device=device)
    if P.scale is not None:
        q = q * P.scale.view(U, 1, 1)
    if P.outlier_mask is not None:
        q = q * P.outlier_mask.view(U, 1, d)
    k, v = _draw_kv(cfg, P, 0, U, 1, g, device)
    return dict(q=q.to(torch.bfloat16), k_new=k[:, 0].to(torch.bfloat16),
                v_new=v[:, 0].to(torch.bfloat16))


def gen_prefill_scorer(cfg: PrefillConfig, device, seed: int = 0):
    """Prefill-scorer inputs: q_win [NL][Hq][w][d], K, V [NL][Hkv][N][d],
    W_O [NL][Hq*d][D] (N(0, wo_std^2)), all bf16."""
    NL, Hq, Hkv, d, N, w = cfg.NL, cfg.Hq, cfg.Hkv, cfg.d, cfg.N, cfg.w
    gq = _gen(device, seed * 7919 + _OFF_PRE_Q)
    q = torch.randn(NL, Hq, w, d, generator=gq, device=device).to(torch.bfloat16)
    gk = _gen(device, seed * 7919 + _OFF_PRE_KV)
    K = torch.empty(NL, Hkv, N, d, dtype=torch.bfloat16, device=device)
    V = torch.empty(NL, Hkv, N, d, dtype=torch.bfloat16, device=device)
    for l in range(NL):
        K[l] = torch.randn(Hkv, N, d, generator=gk, device=device).to(torch.bfloat16)
        V[l] = torch.randn(Hkv, N, d, generator=gk, device=device).to(torch.bfloat16)
    gw = _gen(device, seed * 7919 + _OFF_PRE_W)
    W = torch.empty(NL, Hq * d, cfg.D, dtype=torch.bfloat16, device=device)
    for l in range(NL):
        W[l] = (cfg.wo_std * torch.randn(Hq * d, cfg.D, generator=gw,
                                         device=device)).to(torch.bfloat16)
    return dict(q_win=q, K=K, V=V, W_O=W)
