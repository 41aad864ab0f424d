"""Benchmark of the budgeted-KV decode step on GB300.

Workload (default): the Qwen3-4B attention shape -- batch 16, 36 layers, 32
query / 8 KV heads (4608 units), d = 128, prefill N = 32768, budget L = 3277
slots per KV head, EMA utility (alpha 0.9) refreshed every 8 steps, moment
correction on, fp32 moments.  Step 1 (the one-off pass over N + 1 slots that
evicts down to L) runs untimed-for-the-metric and is reported separately; a
timed step is one steady-state decode step over every unit (append, attention,
head-mean scores, utility refresh on refresh steps, eviction, moment fold,
correction, compaction), i.e. one call of kvc_decode_step.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead (a bounded sample of the same workload on the host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="C2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the sequence count (smaller case for profiling)")
    ap.add_argument("--prefill", type=int, default=None,
                    help="override the prefill length N (smaller case for profiling)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the LaProx prefill scorer (prefill-scoring workload)")
    ap.add_argument("--prefill-layers", type=int, default=None,
                    help="override the layer count of the prefill-scoring workload")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the secondary decode workloads (long context, Llama-3.1-8B, tiny)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ byte model
def step_bytes(cfg, refresh: bool, emit_probs: bool) -> int:
    """Algorithmic HBM bytes of one steady-state step over every unit.

    Per unit: K and V rows of the L slots (the victim's row is read once for
    the moment fold, the new token's row is written), q, k_new, v_new, o, the
    moments (C read + written, means, count), votes when present; on refresh
    steps the utilities (read + written, fp64), positions and the emitted
    fp64 probabilities.  A lazy step without a victim queue (Score-Free, or
    merge mode) reads the utilities and positions for its argmin.  Merge mode
    (KeepKV ZIP-merging) reads the moments without writing them, appends the
    new token, and its merge kernel reads every key row and position once
    more, re-reads the victim and partner rows, writes the merged rows and
    moves the appended slot into the victim's.
    """
    d, G, L = cfg.d, cfg.G, cfg.L
    merge = cfg.merge_recent is not None
    b = 2 * L * d * 2                 # K, V rows read
    b += 2 * d * 2                    # k_new, v_new read
    b += 2 * d * 2                    # new token written (victim slot, or slot L)
    b += G * d * 2                    # q
    b += G * d * 4                    # o
    if merge:
        b += d * d * 4 + 2 * d * 4 + 4    # C, mu_k, mu_v, n read
    else:
        b += 2 * (d * d * 4) + 4 * d * 4 + 8   # C r/w, mu_k / mu_v r/w, n
    b += 16                           # pos / votes / util of the new slot, counts
    if cfg.votes_max or merge:
        b += L * 4
    if refresh:
        b += (L + 1) * 8 * 2 + L * 4  # util r/w, positions
        if emit_probs:
            b += (L + 1) * 8
    elif merge or cfg.T == 0:
        b += L * (8 + 4)              # utilities and positions of the argmin
    if merge:
        b += (L + 1) * (d * 2 + 4)    # merge kernel: key rows and positions
        b += 4 * d * 2 + 2 * d * 2    # victim / partner rows read, merged rows written
        b += 2 * 2 * d * 2 + 32       # appended slot moved (read + write), votes, util
    return b * cfg.U


def fp32_peak_tflops() -> float:
    """CUDA-core fp32 peak of the GPU from its unit counts and the measured
    maximum SM clock: 152 SMs x 128 fp32 lanes x 2 FLOP (FMA) x clock."""
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def mi_flops(cfg) -> int:
    """Algorithmic FLOPs of the moment-informed scores of one steady-state
    step: C (k - mu_k) for every slot of every unit (L + 1 slots, d x d)."""
    return 2 * (cfg.L + 1) * cfg.d * cfg.d * cfg.U


def mi_norm_bytes(cfg) -> int:
    """Algorithmic HBM bytes of the moment-informed residual norms of one
    steady-state step: every slot's key and value row, C, the means, the new
    token, and the norms written and read back by the fused step."""
    d, L = cfg.d, cfg.L
    b = 2 * L * d * 2 + d * d * 4 + 2 * d * 4 + 2 * d * 2 + (L + 1) * 4 * 2
    return b * cfg.U


def prefill_bytes(pc) -> int:
    """Algorithmic HBM bytes of one prefill scoring call: K and V once, the
    window queries, the value-norm factors, the indicator written, then read and
    written by the normalization, read by the four radix passes, the count
    and the write pass, and the keep mask / counts / indices written."""
    M = pc.NL * pc.Hkv * pc.N
    b = 2 * M * pc.d * 2
    b += pc.NL * pc.Hq * pc.w * pc.d * 2
    b += pc.NL * pc.Hkv * pc.d * pc.d * 4
    b += M * 4 * (1 + 2 + 4 + 1 + 1)
    b += M + pc.NL * pc.Hkv * 4 + pc.B_total * 8
    return b


def prefill_flops(pc) -> int:
    """Algorithmic tensor-core FLOPs: q K^T of the G*w window rows once and
    the d x d value-norm factor applied to every v once (the second q K^T pass
    and the three-term split of the factor are implementation choices on
    top)."""
    M = pc.NL * pc.Hkv * pc.N
    return 2 * M * pc.G * pc.w * pc.d + 2 * M * pc.d * pc.d


def run_prefill(pc, dev, reps=5):
    import torch
    from kv_cache_eviction_kvc_gb300 import kvc, workloads as W
    inp = W.gen_prefill_scorer(pc, dev, 0)
    NL, Hq, Hkv, d, N, w, B = pc.NL, pc.Hq, pc.Hkv, pc.d, pc.N, pc.w, pc.B_total
    R = torch.empty(NL, Hkv, d, d, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    kvc.kvc_prefill_prepare(NL, Hq, Hkv, d, pc.D, inp["W_O"], R)
    e1.record(stream)
    torch.cuda.synchronize()
    prep_ms = e0.elapsed_time(e1)
    ws = torch.empty(kvc.kvc_prefill_workspace_size(NL, Hkv, N, B), dtype=torch.uint8, device=dev)
    scores = torch.empty(NL, Hkv, N, dtype=torch.float32, device=dev)
    keep = torch.empty(NL, Hkv, N, dtype=torch.uint8, device=dev)
    counts = torch.empty(NL, Hkv, dtype=torch.int32, device=dev)
    idx = torch.empty(max(B, 1), dtype=torch.int64, device=dev)

    def call(alloc):
        kvc.kvc_prefill_score(NL, Hq, Hkv, d, N, w, B, 1, inp["q_win"], inp["K"], inp["V"], R,
                              scores, keep, counts, idx, ws, alloc=alloc)

    def timed(alloc):
        for _ in range(2):
            call(alloc)
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(alloc)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return sorted(times)[len(times) // 2]
    # the LaProx ablation's other budget allocations: per layer (head-flatten
    # only) and uniform per KV head, same scorer, segmented selection
    alloc_ms = {"head_flatten": timed(kvc.ALLOC_LAYER), "uniform": timed(kvc.ALLOC_HEAD)}
    # MomentKV's SnapKV protocol on the same prompt and budget: accumulated
    # window attention, first-token sink, blocks of 4, per-layer budgets
    snap_keep = torch.empty_like(keep)

    def snap():
        kvc.kvc_prefill_snapkv(NL, Hq, Hkv, d, N, w, B, 4, 1, inp["q_win"], inp["K"], None,
                               snap_keep, None, None, ws)
    snap_ms = median_ms(snap, stream, reps)
    ms = timed(kvc.ALLOC_GLOBAL)
    handoff = run_handoff(pc, inp, keep, dev, stream, reps)
    peak, kind = peaks()
    by = prefill_bytes(pc)
    ach = by / (ms * 1e-3) / 1e9
    fl = prefill_flops(pc)
    return {"workload": pc.name, "description": pc.description, "ms_per_call": ms,
            "calls_per_s": 1000.0 / ms, "prepare_ms": prep_ms,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                         "frac": ach / peak, "peak_kind": kind, "bytes_per_call": by,
                         "algorithmic_tflops": fl / (ms * 1e-3) / 1e12,
                         "kernels": "pack + prefill_attn beside prefill_val + combine + radix select"},
            "kept": int(counts.sum().item()),
            "allocations_ms_per_call": alloc_ms,
            "snapkv_ms_per_call": snap_ms,
            "handoff": handoff}


def median_ms(fn, stream, reps):
    import torch
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return sorted(times)[len(times) // 2]


def run_handoff(pc, inp, keep, dev, stream, reps):
    """The LaProx global selection turned into a decode cache (kept rows
    gathered, a budget per (layer, KV head), the dropped tokens folded into
    the eviction-set moments), timed alone."""
    import torch
    from kv_cache_eviction_kvc_gb300 import kvc
    U, N, d, G = pc.NL * pc.Hkv, pc.N, pc.d, pc.G
    counts = keep.view(U, N).sum(dim=1)
    cap = int(counts.max().item()) + 2
    cap = (cap + 7) // 8 * 8
    from kv_cache_eviction_kvc_gb300.state import DecodeState
    st = DecodeState(U, G, cap, cap - 1, d=d, rule=kvc.RULE_MI, budgets=True, device=dev)
    ws = torch.empty(kvc.kvc_prefill_handoff_workspace_size(U, N), dtype=torch.uint8, device=dev)

    def call():
        kvc.kvc_prefill_handoff(st.params, N, keep, inp["K"], inp["V"], None, None, st.cache,
                                st.moments, st.budget, ws)
    ms = median_ms(call, stream, reps)
    kept = int(counts.sum().item())
    # every prompt row read once (K and V, bf16), the kept rows written once
    by = 2 * U * N * d * 2 + 2 * kept * d * 2
    return {"ms_per_call": ms, "units": U, "cap": cap, "kept": kept,
            "algorithmic_gbs": by / (ms * 1e-3) / 1e9}


def profiled_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of ``kernel`` on the full workload,
    from the ncu capture recorded in profiles/traffic.json, or None when the
    kernel's sources changed since the counters were taken (the record holds
    a hash of those sources)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        with open(fp, "rb") as fh:
            h.update(fh.read())
    return int(rec["traffic_bytes_per_launch"]) if h.hexdigest()[:16] == rec["sha256_16"] else None


# ------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kvc_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------ CPU oracle
def oracle_sample(cfg, seconds: float, max_steps: int | None = None):
    """Time the fp64 oracle on a bounded sample of the steady-state workload:
    Us units whose cache holds L slots, stepping through refresh and lazy
    steps.  Returns (steps/s extrapolated to all units, cores, sample text,
    per-step times)."""
    import numpy as np
    import torch
    from kv_cache_eviction_kvc_gb300 import workloads as W
    from oracle import oracle as O
    cores = len(os.sched_getaffinity(0))
    Us = max(cores, 16)
    small = cfg.with_(B=1, NL=1, Hkv=Us, Hq=Us * cfg.G, N=cfg.L)
    P = W.unit_params(small, "cpu", 0)
    pre = W.gen_prefill(small, "cpu", 0, cap=cfg.L + 1, P=P)
    sess = O.DecodeSession(Us, cfg.G, cfg.d, cfg.L + 64)
    for u in range(Us):
        sess.load(u, pre["K"][u, : cfg.L], pre["V"][u, : cfg.L],
                  None if pre["votes"] is None else pre["votes"][u, : cfg.L].numpy())
    times = []
    t = 0
    t_start = time.perf_counter()
    while True:
        t += 1
        inp = W.gen_step(small, "cpu", t, 0, P)
        t0 = time.perf_counter()
        O.decode_step(sess, t, cfg.L + t - 1, inp["q"], inp["k_new"], inp["v_new"], L=cfg.L,
                      rule=cfg.rule, alpha=cfg.alpha, T=cfg.T, correction=cfg.correction,
                      merge_recent=cfg.merge_recent)
        times.append(time.perf_counter() - t0)
        if max_steps is not None and t >= max_steps:
            break
        if max_steps is None and (time.perf_counter() - t_start > seconds or t >= 40):
            break
    sess.close()
    per_unit_step = sum(times) / (len(times) * Us)
    rate = 1.0 / (per_unit_step * cfg.U)
    sample = (f"{Us} units x {len(times)} steady-state steps of this workload (L={cfg.L}, "
              f"T={cfg.T}) on the fp64 oracle, OpenMP over units; steps/s scaled by "
              f"{Us}/{cfg.U} units")
    return rate, cores, sample, times


# ------------------------------------------------------------ GPU arm
def is_refresh(t, T):
    """Refresh steps: t = 1 and every T-th step after it; T = 0: step 1 only."""
    return t == 1 if T == 0 else (T == 1 or (t - 1) % T == 0)


def run_ours(args, cfg, rank, world, steps=None, warmup=None, e2e=True, sample_clocks=True):
    """Step 1, then W warm-up and K timed steady-state steps of kvc_decode_step
    over every unit of ``cfg``; returns the JSON record."""
    import torch
    from kv_cache_eviction_kvc_gb300 import kvc, workloads as W
    from kv_cache_eviction_kvc_gb300.state import DecodeState

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    kvc.load()
    seed = rank
    U, G, N, L = cfg.U, cfg.G, cfg.N, cfg.L
    P = W.unit_params(cfg, dev, seed)
    merge = cfg.merge_recent is not None
    mi = cfg.rule == W.RULE_MI
    chained = cfg.rule == W.RULE_EMA_CHAINED
    st = DecodeState(U, G, N + 1, L, rule=cfg.rule, alpha=cfg.alpha, refresh_period=cfg.T,
                     correction=cfg.correction, votes=bool(cfg.votes_max) or merge,
                     kmax=N + 1 - L, device=dev, merge_recent=cfg.merge_recent,
                     chain=(cfg.NL, cfg.Hkv) if chained else None)
    # the prefill is drawn straight into the state's K / V (no second copy)
    pre = W.gen_prefill(cfg, dev, seed, cap=N + 1, P=P, out_K=st.K, out_V=st.V)
    st.load_prefill(pre["K"], pre["V"], pre["votes"], pre["pos"], pre["len"])
    del pre
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream(dev)

    # step 1: the one-off pass over N + 1 slots (general path), under the
    # workload's first-step rule where it has one (the moment-informed
    # workload compresses the prompt by attention first; every token this
    # removes is folded into the moments)
    inp = W.gen_step(cfg, dev, 1, seed, P)
    if cfg.first_rule is not None:
        st.params.rule = cfg.first_rule
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st.step(1, N, inp["q"], inp["k_new"], inp["v_new"], max_len=N + 1)
    e1.record(stream)
    torch.cuda.synchronize()
    step1_ms = e0.elapsed_time(e1)
    st.params.rule = cfg.rule
    assert st.device_status() == 0
    st.set_kmax(1)

    total = warmup + steps
    inputs = [W.gen_step(cfg, dev, 2 + i, seed, P) for i in range(total)]
    torch.cuda.synchronize()
    launches = 0
    # moment-informed rule: the residual-norm kernel, then the fused step;
    # merge mode: the fused step, then the merge kernel; the layer-chained EMA
    # takes the five-call sequence (attend in two kernels, the per-sequence
    # aggregation, fold, correction, compaction)
    per_step_launches = 6 if chained else (2 if (mi or merge) else 1)

    def do_step(t, x, events=None, o=None):
        nonlocal launches
        if events is not None:
            events[0].record(stream)
        st.step(t, N + t - 1, x["q"], x["k_new"], x["v_new"], max_len=L + 1, o=o)
        if events is not None:
            events[1].record(stream)
        launches += per_step_launches

    for i in range(warmup):
        do_step(2 + i, inputs[i])
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if sample_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    launches = 0
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(steps):
        do_step(2 + warmup + k, inputs[warmup + k], ev[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    timed_launches = launches
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [a.elapsed_time(b) for a, b in ev]
    if world > 1:
        from kv_cache_eviction_kvc_gb300.dist import max_over_ranks
        total_ms = max_over_ranks(total_ms, dev)
    assert st.device_status() == 0

    # algorithmic bytes of the timed launches (refresh pattern of steps 2 + i)
    steps_t = [2 + warmup + k for k in range(steps)]
    ref_flags = [is_refresh(t, cfg.T) for t in steps_t]
    bytes_list = [step_bytes(cfg, r, True) for r in ref_flags]
    avg_bytes = sum(bytes_list) / len(bytes_list)
    avg_launch_ms = sum(per_launch) / len(per_launch)
    achieved = avg_bytes / (avg_launch_ms * 1e-3) / 1e9
    lazy = [ms for ms, r in zip(per_launch, ref_flags) if not r]
    refr = [ms for ms, r in zip(per_launch, ref_flags) if r]
    lazy_ms = statistics.median(lazy) if lazy else None
    refresh_ms = statistics.median(refr) if refr else None
    # steady state weighted by the refresh period: one refresh step in T
    if cfg.T >= 2 and lazy_ms is not None and refresh_ms is not None:
        steady_ms = (refresh_ms + (cfg.T - 1) * lazy_ms) / cfg.T
        steady_bytes = (step_bytes(cfg, True, True) + (cfg.T - 1) * step_bytes(cfg, False, True)) / cfg.T
    else:
        steady_ms = lazy_ms if (cfg.T == 0 and lazy_ms is not None) else statistics.median(per_launch)
        steady_bytes = step_bytes(cfg, cfg.T == 1, True)

    # end to end through host buffers: every step copies its inputs from
    # pinned host memory and its output o back.  Two copy streams (one per
    # direction) and double-buffered device inputs / outputs let the copies of
    # step k + 1 / k - 1 overlap the compute of step k, as a serving loop would.
    # The window has as many steps as the timed one and starts at the same
    # step index modulo T, so both hold the same mix of refresh and lazy steps.
    e2e_rec = None
    if e2e:
        nE = steps
        t_next = 2 + total
        t0 = 2 + warmup
        if cfg.T >= 2:
            pad = (t0 - t_next) % cfg.T
        else:
            pad = 0
        extra = [W.gen_step(cfg, dev, t_next + i, seed, P) for i in range(pad)]
        for i in range(pad):                       # untimed: align the refresh phase
            do_step(t_next + i, extra[i])
        base_t = t_next + pad
        names = ("q", "k_new", "v_new")
        host_in = []
        for j in range(nE):
            x = W.gen_step(cfg, dev, base_t + j, seed, P)
            host_in.append({k: x[k].cpu().pin_memory() for k in names})
        din = [{k: torch.empty_like(inputs[0][k]) for k in names} for _ in range(2)]
        dout = [torch.empty_like(st.o) for _ in range(2)]
        o_host = [torch.empty(st.o.shape, dtype=st.o.dtype).pin_memory() for _ in range(2)]
        hs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nE)]
        ev_done = [torch.cuda.Event() for _ in range(nE)]
        ev_out = [torch.cuda.Event() for _ in range(nE)]
        torch.cuda.synchronize()

        def h2d(j):
            with torch.cuda.stream(hs):
                if j >= 2:
                    hs.wait_event(ev_done[j - 2])          # buffer read by step j - 2
                for k in names:
                    din[j % 2][k].copy_(host_in[j][k], non_blocking=True)
                ev_in[j].record(hs)

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        hs.wait_stream(stream)
        ds.wait_stream(stream)
        h2d(0)
        for j in range(nE):
            if j + 1 < nE:
                h2d(j + 1)
            stream.wait_event(ev_in[j])
            if j >= 2:
                stream.wait_event(ev_out[j - 2])           # o buffer read back
            do_step(base_t + j, din[j % 2], o=dout[j % 2])
            ev_done[j].record(stream)
            with torch.cuda.stream(ds):
                ds.wait_event(ev_done[j])
                o_host[j % 2].copy_(dout[j % 2], non_blocking=True)
                ev_out[j].record(ds)
        stream.wait_stream(ds)
        stream.wait_stream(hs)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / nE
        if world > 1:
            from kv_cache_eviction_kvc_gb300.dist import max_over_ranks
            e2e_ms = max_over_ranks(e2e_ms, dev)
        bi = sum(v.numel() * v.element_size() for v in host_in[0].values())
        bo = o_host[0].numel() * o_host[0].element_size()
        e2e_rec = {"value": world * 1000.0 / e2e_ms, "unit": UNIT, "h2d_bytes_per_step": bi,
                   "d2h_bytes_per_step": bo, "steps": nE,
                   "first_step": base_t,
                   "note": "inputs H2D from pinned memory and o D2H every step, on two copy "
                           "streams overlapping the compute stream; same step count and "
                           "refresh phase as the timed window"}
        assert st.device_status() == 0

    peak, peak_kind = peaks()
    ms_per_step = total_ms / steps
    kname = ("fused_step_kernel + zip_merge_kernel (kvc_decode_step, merge mode)"
             if merge else
             "attend_chunk + attend_final + aggregate_chained + moment_fold + correct + "
             "compact (kvc_decode_step, layer-chained EMA)" if chained else
             "fused_step_kernel (kvc_decode_step, steady state)")
    traffic = None
    if (not merge and not mi and args.batch is None and args.prefill is None
            and cfg.T >= 1 and args.config == "C2" and cfg.name == W.C2.name):
        tr_lazy = profiled_traffic("fused_step_kernel_qwen3-4b_lazy")
        tr_ref = profiled_traffic("fused_step_kernel_qwen3-4b_refresh")
        if tr_lazy is not None and tr_ref is not None:
            nr = sum(ref_flags)
            traffic = (nr * tr_ref + (steps - nr) * tr_lazy) / steps
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "traffic_note": "ncu dram read+write per launch (profiles/traffic.json), "
                                "averaged over the window's refresh / lazy mix; null when "
                                "the kernel changed since the capture",
                "peak_kind": peak_kind, "kernel": kname,
                "bytes_per_launch": avg_bytes, "avg_launch_ms": avg_launch_ms}
    if mi:
        # the moment-informed step streams the cache twice: the residual-norm
        # kernel (keys through the tensor cores, values on CUDA cores), then
        # the fused step scoring alpha ||r||
        mb = avg_bytes + mi_norm_bytes(cfg)
        ach = mb / (avg_launch_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                    "frac": ach / peak, "traffic": None, "peak_kind": peak_kind,
                    "kernel": "mi_norm_kernel (tcgen05) + fused_step_kernel (kvc_decode_step, "
                              "rule MI, steady state)",
                    "bytes_per_launch": mb, "avg_launch_ms": avg_launch_ms,
                    "contraction_tflops": mi_flops(cfg) / (avg_launch_ms * 1e-3) / 1e12,
                    "contraction_flops_per_step": mi_flops(cfg)}
        achieved = ach
    value = world * steps / (total_ms * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 K/V/q, fp32 accumulate and moments, fp64 utilities",
        "data": "synthetic (seeded K/V 64-centre mixtures; no model weights)",
        "config": {"workload": cfg.name, "description": cfg.description, "units": cfg.U,
                   "budget_L": L, "prefill_N": N, "refresh_period": cfg.T,
                   "merge_recent": cfg.merge_recent,
                   "alpha": cfg.alpha, "parallelism": f"replicas x{world} (independent units)",
                   "l2": "inputs larger than L2: %.2f GB of HBM traffic per step" % (avg_bytes / 1e9)
                         if avg_bytes > 129e6 else
                         "working set %.1f MB fits L2: launch-bound, no flush" % (avg_bytes / 1e6)},
        "achieved_gbs": achieved,
        "hbm_frac": achieved / peak,
        "step1_ms": step1_ms,
        "lazy_ms": lazy_ms,
        "refresh_ms": refresh_ms,
        "refresh_steps_in_window": sum(ref_flags),
        "steady_state": {"ms_per_step": steady_ms, "steps_per_s": world * 1000.0 / steady_ms,
                         "hbm_frac": steady_bytes / (steady_ms * 1e-3) / 1e9 / peak,
                         "note": "one refresh step in T (median refresh and lazy launch times)"},
        "roofline": roofline,
        "clocks": clocks,
        "gpu_launches": timed_launches,
        "e2e": e2e_rec,
    }
    del st, inputs
    torch.cuda.empty_cache()
    return res


def summary(rec):
    """The figures of a secondary workload's line."""
    keys = ("value", "unit", "ms_per_step", "step1_ms", "lazy_ms", "refresh_ms",
            "achieved_gbs", "hbm_frac", "steady_state", "gpu_launches")
    out = {k: rec[k] for k in keys if k in rec}
    out["config"] = rec["config"]
    out["roofline_frac"] = rec["roofline"]["frac"]
    out["clocks"] = rec["clocks"]
    return out


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    from kv_cache_eviction_kvc_gb300 import workloads as W
    cfg = W.DECODE_CONFIGS[args.config]
    if args.prefill_only:
        import torch
        pc = W.C3 if args.prefill_layers is None else W.C3.with_(NL=args.prefill_layers)
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"metric": "prefill scoring calls/sec", **run_prefill(pc, dev)}))
        return
    if args.batch is not None:
        cfg = cfg.with_(B=args.batch, name=cfg.name + f"-b{args.batch}")
    if args.prefill is not None:
        cfg = cfg.with_(N=args.prefill, name=cfg.name + f"-n{args.prefill}")
    if args.impl == "reference":
        if rank != 0:
            return
        rate_steps = []
        cores = len(os.sched_getaffinity(0))
        budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
        rate, cores, sample, times = oracle_sample(cfg, budget, max_steps=args.warmup + args.steps + 1)
        times = times[1 + args.warmup:] or times
        Us = max(cores, 16)
        per = sum(times) / len(times)
        value = 1.0 / (per / Us * cfg.U)
        res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
               "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 / value,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "f64", "data": "synthetic",
               "config": {"workload": cfg.name, "description": cfg.description},
               "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample},
               "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res = run_ours(args, cfg, rank, world)
    if rank == 0 and not args.no_prefill and args.batch is None and args.prefill is None:
        import torch
        torch.cuda.empty_cache()
        res["prefill"] = run_prefill(W.C3, torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
    if not args.no_extra and args.batch is None and args.prefill is None and args.config == "C2":
        # the other decode workloads at 1 GPU (every rank runs its replica)
        res["other_workloads"] = {}
        for name in ("C4", "C1", "C0"):
            try:
                rec = run_ours(args, W.DECODE_CONFIGS[name], rank, world,
                               steps=max(args.steps, 20), warmup=max(args.warmup, 3),
                               e2e=False, sample_clocks=(name == "C4"))
                res["other_workloads"][name] = summary(rec)
            except Exception as exc:      # a secondary line never sinks the main one
                res["other_workloads"][name] = {"error": f"{type(exc).__name__}: {exc}"}
    if rank == 0:
        if not args.no_cpu_baseline:
            rate, cores, sample, _ = oracle_sample(cfg, args.cpu_seconds)
            res["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                   "sample": sample}
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
