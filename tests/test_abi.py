"""The C-ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching a
device (these calls need no GPU)."""
import ctypes
import os
import re

import pytest

from kv_cache_eviction_kvc_gb300 import kvc as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    return re.findall(r"^KVC_API\s+[\w\s\*]+?\b(kvc_\w+)\s*\(", src, flags=re.M)


def test_library_exports_every_declared_symbol():
    lib = K.load()
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(K.EXPORTED)


def test_version_matches_header():
    src = open(os.path.join(ROOT, "include", "kvc.h")).read()
    v = int(re.search(r"#define KVC_VERSION (\d+)", src).group(1))
    assert K.kvc_version() == v
    assert K.kvc_status_string(0) == "KVC_OK"
    assert K.kvc_status_string(6) == "KVC_ERR_WORKSPACE"


def test_workspace_size_host_only():
    p = K.make_params(U=4, G=4, cap=100, L=10)
    n = K.kvc_decode_workspace_size(p)
    # status + logits + split partials + lengths + queues + scratch
    assert n >= 4 * 4 * 100 * 4 + 4 * 1 * 4 * 130 * 4
    assert K.kvc_decode_workspace_size(K.make_params(U=4, G=3, cap=100, L=10)) == 0


def _lib_call_attend(p, **kw):
    lib = K.load()
    cache = K.kvc_cache(*(kw.get(k, 16 * (i + 1)) for i, k in enumerate(["K", "V", "votes", "pos", "util", "len"])))
    ws = kw.get("ws", 256)
    return lib.kvc_decode_attend(ctypes.byref(p), kw.get("t", 1), 0, kw.get("max_len", 5),
                                 16, 16, 16, ctypes.byref(cache), 16, 16, None,
                                 ws, kw.get("ws_bytes", 1 << 40), None)


@pytest.mark.parametrize("field,value,code", [
    ("d", 64, 5), ("G", 3, 5), ("U", 0, 1), ("L", 0, 1), ("L", 100, 1),
    ("refresh_period", -1, 1), ("refresh_period", 11, 1), ("rule", 7, 1),
    ("alpha", 1.0, 1), ("correction", 3, 1), ("cap", 0, 5)])
def test_bad_params_rejected_on_host(field, value, code):
    p = K.make_params(U=2, G=4, cap=100, L=10)
    setattr(p, field, value)
    assert _lib_call_attend(p) == code
    assert K.kvc_last_error() != ""


def test_bad_buffers_rejected_on_host():
    p = K.make_params(U=2, G=4, cap=100, L=10)
    assert _lib_call_attend(p, K=None) == 1                 # null cache pointer
    assert _lib_call_attend(p, K=18) == 1                   # misaligned K
    assert _lib_call_attend(p, ws=None) == 6                # no workspace
    assert _lib_call_attend(p, ws=128) == 6                 # misaligned workspace
    assert _lib_call_attend(p, ws_bytes=16) == 6            # too small
    assert _lib_call_attend(p, max_len=101) == 2            # beyond capacity
    assert _lib_call_attend(p, t=0) == 1                    # steps are 1-based
    assert "workspace" in K.kvc_last_error() or "t =" in K.kvc_last_error()


def test_binding_refuses_host_tensors():
    import torch
    p = K.make_params(U=1, G=4, cap=8, L=4)
    with pytest.raises(ValueError):
        K.kvc_decode_workspace_init(p, torch.zeros(16, dtype=torch.uint8))


@pytest.mark.parametrize("field,value", [
    ("merge", 2), ("merge_recent", -1), ("rule", 4)])
def test_bad_extension_params_rejected_on_host(field, value):
    """ZIP-merging and moment-informed parameters are validated before any
    launch."""
    p = K.make_params(U=2, G=4, cap=100, L=10)
    setattr(p, field, value)
    assert _lib_call_attend(p) == 1
    assert K.kvc_last_error() != ""


def test_moment_informed_rule_needs_refresh_every_step():
    # (every call in this file is refused before a launch: the pointers are fake)
    p = K.make_params(U=2, G=4, cap=100, L=10, rule=K.RULE_MI, refresh_period=4)
    assert _lib_call_attend(p) == 1
    assert "refresh period" in K.kvc_last_error()


def test_zip_merge_needs_votes():
    """Merged slots carry p_e + p_c: kvc_zip_merge refuses a cache without
    votes (host check, no launch)."""
    lib = K.load()
    p = K.make_params(U=2, G=4, cap=100, L=10, merge_recent=4)
    cache = K.kvc_cache(16, 32, None, 64, 128, 256)
    rc = lib.kvc_zip_merge(ctypes.byref(p), 5, 16, ctypes.byref(cache), 1, 16, 16, None,
                           256, 1 << 40, None)
    assert rc == 1 and "votes" in K.kvc_last_error()


def test_prefill_allocation_arguments_checked_on_host():
    """An unknown allocation, or a budget that does not divide into the
    allocation's segments, is refused before any pointer is touched."""
    lib = K.load()
    args = [None] * 10
    rc = lib.kvc_prefill_score(2, 8, 2, 128, 64, 8, 12, 1, 5, *args[:8], None, 0, None)
    assert rc == 1 and "alloc" in K.kvc_last_error()
    rc = lib.kvc_prefill_score(2, 8, 2, 128, 64, 8, 6, 1, K.ALLOC_HEAD, *args[:8], None, 0, None)
    assert rc == 1 and "multiple" in K.kvc_last_error()


def _lib_call_attend_noalloc(p, **kw):
    lib = K.load()
    cache = K.kvc_cache(*(kw.get(k, 16 * (i + 1)) for i, k in enumerate(["K", "V", "votes", "pos", "util", "len"])))
    return lib.kvc_decode_attend_noalloc(ctypes.byref(p), kw.get("t", 1), 0, kw.get("max_len", 5),
                                         16, 16, 16, ctypes.byref(cache), 16, 16, None, None, None)


@pytest.mark.parametrize("field,value", [
    ("d", 64), ("G", 3), ("U", 0), ("L", 0), ("L", 100), ("refresh_period", 11),
    ("rule", 7), ("alpha", 1.0), ("correction", 3), ("cap", 0), ("cap", 1 << 20),
    ("merge", 2), ("merge_recent", -1)])
def test_noalloc_rejects_what_attend_rejects(field, value):
    """The entry point without a workspace validates its parameters exactly as
    kvc_decode_attend does: the same status code for every rejected field
    (host checks only; the pointers are fake and nothing launches)."""
    p = K.make_params(U=2, G=4, cap=100, L=10)
    setattr(p, field, value)
    code = _lib_call_attend(p)
    assert code != 0
    assert _lib_call_attend_noalloc(p) == code
    assert K.kvc_last_error() != ""


def test_noalloc_rejects_bad_buffers_like_attend():
    p = K.make_params(U=2, G=4, cap=100, L=10)
    for kw in ({"K": None}, {"K": 18}, {"max_len": 101}, {"t": 0}):
        assert _lib_call_attend_noalloc(p, **kw) == _lib_call_attend(p, **kw) != 0


def test_long_moment_informed_first_step_refused_on_host():
    """MomentKV's loop re-scores the whole cache after every fold: a step
    that would remove thousands of slots from a long prompt is refused
    before any launch (KVC_ERR_UNSUPPORTED), by kvc_decode_step and by
    kvc_mi_evict alike; a combination of the rule with merging is invalid."""
    lib = K.load()
    p = K.make_params(U=2, G=4, cap=40000, L=100, rule=K.RULE_MI, refresh_period=1)
    cache = K.kvc_cache(16, 32, None, 64, 128, 256)
    mom = K.kvc_moments(16, 32, 64, 128)
    rc = lib.kvc_decode_step(ctypes.byref(p), 1, 0, 32769, 16, 16, 16, ctypes.byref(cache),
                             ctypes.byref(mom), 16, None, 40000, 16, None, 16, 256, 1 << 40, None)
    assert rc == 5 and "rounds" in K.kvc_last_error()
    rc = lib.kvc_mi_evict(ctypes.byref(p), 32769, ctypes.byref(cache), ctypes.byref(mom), 16,
                          40000, 16, None, 16, 256, 1 << 40, None)
    assert rc == 5
    p2 = K.make_params(U=2, G=4, cap=100, L=10, rule=K.RULE_MI, refresh_period=1, merge_recent=4)
    assert _lib_call_attend(p2) == 1 and "merging" in K.kvc_last_error()
