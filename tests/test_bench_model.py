"""The byte and FLOP models behind bench.py's roofline figures, pinned to
the values the profiles quote and to their term-by-term definitions."""
import json
import os

import pytest

import bench
from kv_cache_eviction_kvc_gb300 import workloads as W


def test_lazy_step_bytes_of_the_decode_workload():
    """K and V of L slots, new token, q, o, moments r/w: 8.364 GB per lazy
    launch over 4608 units (the figure the fused-kernel profile scales the
    ncu traffic against)."""
    assert bench.step_bytes(W.C2, refresh=False, emit_probs=True) == 8363814912


def test_refresh_step_adds_utilities_positions_and_probabilities():
    L, U = W.C2.L, W.C2.U
    extra = bench.step_bytes(W.C2, True, True) - bench.step_bytes(W.C2, False, True)
    assert extra == U * ((L + 1) * 16 + L * 4 + (L + 1) * 8)


def test_score_free_lazy_step_reads_the_argmin_inputs():
    L, U = W.C2.L, W.C2.U
    d = bench.step_bytes(W.C2_SCORE_FREE, False, True) - bench.step_bytes(W.C2, False, True)
    assert d == U * L * (8 + 4)


def test_merge_mode_bytes():
    """Moments read only (no write-back), votes, the argmin inputs and the
    merge kernel's pass over the key rows and positions."""
    cfg, L, U, dd = W.C2_ZIP, W.C2.L, W.C2.U, W.C2.d
    base = bench.step_bytes(W.C2, False, True) // U
    got = bench.step_bytes(cfg, False, True) // U
    moments_saved = (2 * dd * dd * 4 + 4 * dd * 4 + 8) - (dd * dd * 4 + 2 * dd * 4 + 4)
    added = L * 4 + L * 12 + (L + 1) * (dd * 2 + 4) + 4 * dd * 2 + 2 * dd * 2 + 2 * 2 * dd * 2 + 32
    assert got == base - moments_saved + added


def test_moment_informed_flops_and_fp32_peak():
    assert bench.mi_flops(W.C2_MI) == 2 * 3278 * 128 * 128 * 4608 == 494961426432
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    mhz = 2070.0
    if os.path.exists(path):
        mhz = float(json.load(open(path)).get("sm_max_mhz", mhz))
    assert bench.fp32_peak_tflops() == pytest.approx(152 * 128 * 2 * mhz * 1e6 / 1e12)


def test_moment_informed_norm_bytes():
    """Keys and values of L slots, C, the two means, the new token, the norms
    written then read by the fused step, per unit."""
    d, L, U = 128, 3277, 4608
    per = 2 * L * d * 2 + d * d * 4 + 2 * d * 4 + 2 * d * 2 + (L + 1) * 8
    assert bench.mi_norm_bytes(W.C2_MI) == per * U
