"""Thin ctypes binding of libkvc (the C ABI declared in ``include/kvc.h``).

Argument marshalling only: every function takes torch tensors (device
memory), checks dtype / device / contiguity, passes raw pointers to the
library function of the same name and raises :class:`KvcError` on a non-OK
status.  All arithmetic runs in the CUDA kernels of libkvc; there is no
fallback.  If the library cannot be built or loaded, importing the binding
fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

KVC_OK = 0
STATUS_NAMES = {0: "KVC_OK", 1: "KVC_ERR_INVALID_ARG", 2: "KVC_ERR_SHAPE",
                3: "KVC_ERR_CUDA", 4: "KVC_ERR_TIMEOUT", 5: "KVC_ERR_UNSUPPORTED",
                6: "KVC_ERR_WORKSPACE"}
RULE_SINGLE, RULE_CUMULATIVE, RULE_EMA, RULE_MI, RULE_EMA_CHAINED = 0, 1, 2, 3, 4
CORR_OFF, CORR_ZERO_ORDER, CORR_FIRST_ORDER = 0, 1, 2
ALLOC_GLOBAL, ALLOC_LAYER, ALLOC_HEAD = 0, 1, 2

EXPORTED = (
    "kvc_version", "kvc_last_error", "kvc_status_string",
    "kvc_decode_workspace_size", "kvc_decode_workspace_init", "kvc_get_device_status",
    "kvc_decode_attend", "kvc_aggregate_evict", "kvc_moment_update", "kvc_correct",
    "kvc_compact", "kvc_zip_merge", "kvc_mi_scores", "kvc_mi_evict", "kvc_decode_step", "kvc_decode_attend_noalloc", "kvc_prefill_prepare",
    "kvc_prefill_workspace_size", "kvc_prefill_score", "kvc_prefill_window_attention",
    "kvc_prefill_snapkv", "kvc_prefill_handoff_workspace_size", "kvc_prefill_handoff",
)


class KvcError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class kvc_params(ctypes.Structure):
    _fields_ = [("U", ctypes.c_int32), ("G", ctypes.c_int32), ("d", ctypes.c_int32),
                ("cap", ctypes.c_int32), ("L", ctypes.c_int32), ("rule", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("refresh_period", ctypes.c_int32),
                ("correction", ctypes.c_int32), ("merge", ctypes.c_int32),
                ("merge_recent", ctypes.c_int32), ("budget", ctypes.c_void_p),
                ("chain_layers", ctypes.c_int32), ("chain_heads", ctypes.c_int32)]


class kvc_cache(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("votes", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("util", ctypes.c_void_p), ("len", ctypes.c_void_p)]


class kvc_moments(ctypes.Structure):
    _fields_ = [("n", ctypes.c_void_p), ("mu_k", ctypes.c_void_p),
                ("mu_v", ctypes.c_void_p), ("C", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build: bool = True):
    """Load libkvc (building it first when sources changed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build else _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libkvc not built at {path}")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    PP = ctypes.POINTER(kvc_params)
    PC = ctypes.POINTER(kvc_cache)
    PM = ctypes.POINTER(kvc_moments)
    sigs = {
        "kvc_version": (I32, []),
        "kvc_last_error": (ctypes.c_char_p, []),
        "kvc_status_string": (ctypes.c_char_p, [I32]),
        "kvc_decode_workspace_size": (SZ, [PP]),
        "kvc_decode_workspace_init": (I32, [PP, P, SZ, P]),
        "kvc_get_device_status": (I32, [P, SZ, P, ctypes.POINTER(I32)]),
        "kvc_decode_attend": (I32, [PP, I32, I32, I32, P, P, P, PC, P, P, P, P, SZ, P]),
        "kvc_aggregate_evict": (I32, [PP, I32, P, PC, I32, P, P, P, P, SZ, P]),
        "kvc_moment_update": (I32, [PP, PC, I32, P, P, PM, P, SZ, P]),
        "kvc_correct": (I32, [PP, P, PC, I32, P, P, P, P, PM, P, P, P, P, SZ, P]),
        "kvc_compact": (I32, [PP, PC, I32, P, P, P, SZ, P]),
        "kvc_zip_merge": (I32, [PP, I32, P, PC, I32, P, P, P, P, SZ, P]),
        "kvc_mi_scores": (I32, [PP, PC, PM, I32, P, P, P]),
        "kvc_mi_evict": (I32, [PP, I32, PC, PM, P, I32, P, P, P, P, SZ, P]),
        "kvc_decode_step": (I32, [PP, I32, I32, I32, P, P, P, PC, PM, P, P, I32, P, P, P, P, SZ, P]),
        "kvc_decode_attend_noalloc": (I32, [PP, I32, I32, I32, P, P, P, PC, P, P, P, P, P]),
        "kvc_prefill_prepare": (I32, [I32, I32, I32, I32, I32, P, P, P]),
        "kvc_prefill_workspace_size": (SZ, [I32, I32, I32, I64]),
        "kvc_prefill_score": (I32, [I32, I32, I32, I32, I32, I32, I64, I32, I32, P, P, P, P, P,
                                    P, P, P, P, SZ, P]),
        "kvc_prefill_window_attention": (I32, [I32, I32, I32, I32, I32, I32, P, P, P, P, P, SZ,
                                               P]),
        "kvc_prefill_handoff_workspace_size": (SZ, [I32, I32]),
        "kvc_prefill_handoff": (I32, [PP, I32, P, P, P, P, P, PC, PM, P, P, SZ, P]),
        "kvc_prefill_snapkv": (I32, [I32, I32, I32, I32, I32, I32, I64, I32, I32, P, P, P, P, P,
                                     P, P, SZ, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != KVC_OK:
        raise KvcError(status, load().kvc_last_error().decode())


def _ptr(t, dtype=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_params(U, G, cap, L, rule=RULE_EMA, alpha=0.9, refresh_period=1,
                correction=CORR_FIRST_ORDER, d=128, merge_recent=None, budget=None,
                chain=None) -> kvc_params:
    """merge_recent = R (not None) turns on KeepKV ZIP-merging with the last R
    positions excluded from the partner search; budget (a device int32 [U]
    tensor, kept alive by the caller) gives every unit its own budget;
    chain = (NL, Hkv) groups the units by sequence for the layer-chained EMA."""
    merge = 0 if merge_recent is None else 1
    NL, Hkv = (0, 0) if chain is None else (int(chain[0]), int(chain[1]))
    return kvc_params(U, G, d, cap, L, rule, alpha, refresh_period, correction, merge,
                      0 if merge_recent is None else int(merge_recent),
                      _ptr(budget, torch.int32, "budget", optional=True), NL, Hkv)


def make_cache(K, V, votes, pos, util, length) -> kvc_cache:
    return kvc_cache(_ptr(K, torch.bfloat16, "K"), _ptr(V, torch.bfloat16, "V"),
                     _ptr(votes, torch.int32, "votes", optional=True),
                     _ptr(pos, torch.int32, "pos"), _ptr(util, torch.float64, "util"),
                     _ptr(length, torch.int32, "len"))


def make_moments(n, mu_k, mu_v, C) -> kvc_moments:
    return kvc_moments(_ptr(n, torch.float32, "n"), _ptr(mu_k, torch.float32, "mu_k"),
                       _ptr(mu_v, torch.float32, "mu_v"), _ptr(C, torch.float32, "C"))


# ------------------------------------------------------------------ library

def kvc_version() -> int:
    return int(load().kvc_version())


def kvc_last_error() -> str:
    return load().kvc_last_error().decode()


def kvc_status_string(status: int) -> str:
    return load().kvc_status_string(int(status)).decode()


# ------------------------------------------------------------------ decode

def kvc_decode_workspace_size(p: kvc_params) -> int:
    return int(load().kvc_decode_workspace_size(ctypes.byref(p)))


def kvc_decode_workspace_init(p: kvc_params, ws: torch.Tensor, stream=None):
    _check(load().kvc_decode_workspace_init(ctypes.byref(p), _ptr(ws, torch.uint8, "ws"),
                                            ws.numel(), _stream(stream)))


def kvc_get_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(load().kvc_get_device_status(_ptr(ws, torch.uint8, "ws"), ws.numel(),
                                        _stream(stream), ctypes.byref(out)))
    return int(out.value)


def kvc_decode_attend(p, t, new_pos, max_len, q, k_new, v_new, cache: kvc_cache, lse, f_all,
                      probs, ws, stream=None):
    bf = torch.bfloat16
    _check(load().kvc_decode_attend(
        ctypes.byref(p), int(t), int(new_pos), int(max_len), _ptr(q, bf, "q"),
        _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"), ctypes.byref(cache),
        _ptr(lse, torch.float32, "lse"), _ptr(f_all, torch.float32, "f_all"),
        _ptr(probs, torch.float64, "probs", optional=True), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(stream)))


def kvc_aggregate_evict(p, t, probs, cache: kvc_cache, kmax, evict_idx, evict_pos, n_evict, ws,
                        stream=None):
    i32 = torch.int32
    _check(load().kvc_aggregate_evict(
        ctypes.byref(p), int(t), _ptr(probs, torch.float64, "probs", optional=True),
        ctypes.byref(cache), int(kmax), _ptr(evict_idx, i32, "evict_idx"),
        _ptr(evict_pos, i32, "evict_pos", optional=True), _ptr(n_evict, i32, "n_evict"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def kvc_moment_update(p, cache: kvc_cache, kmax, evict_idx, n_evict, mom: kvc_moments, ws,
                      stream=None):
    i32 = torch.int32
    _check(load().kvc_moment_update(
        ctypes.byref(p), ctypes.byref(cache), int(kmax), _ptr(evict_idx, i32, "evict_idx"),
        _ptr(n_evict, i32, "n_evict"), ctypes.byref(mom), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(stream)))


def kvc_correct(p, q, cache: kvc_cache, kmax, evict_idx, n_evict, lse, f_all, mom: kvc_moments,
                o, f_R, logZ_R, ws, stream=None):
    i32, f32 = torch.int32, torch.float32
    _check(load().kvc_correct(
        ctypes.byref(p), _ptr(q, torch.bfloat16, "q"), ctypes.byref(cache), int(kmax),
        _ptr(evict_idx, i32, "evict_idx"), _ptr(n_evict, i32, "n_evict"),
        _ptr(lse, f32, "lse"), _ptr(f_all, f32, "f_all"), ctypes.byref(mom),
        _ptr(o, f32, "o"), _ptr(f_R, f32, "f_R", optional=True),
        _ptr(logZ_R, f32, "logZ_R", optional=True), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)))


def kvc_compact(p, cache: kvc_cache, kmax, evict_idx, n_evict, ws, stream=None):
    i32 = torch.int32
    _check(load().kvc_compact(
        ctypes.byref(p), ctypes.byref(cache), int(kmax), _ptr(evict_idx, i32, "evict_idx"),
        _ptr(n_evict, i32, "n_evict"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)))


def kvc_mi_scores(p, cache: kvc_cache, mom: kvc_moments, max_len, probs, scores, stream=None):
    f64 = torch.float64
    _check(load().kvc_mi_scores(
        ctypes.byref(p), ctypes.byref(cache), ctypes.byref(mom), int(max_len),
        _ptr(probs, f64, "probs"), _ptr(scores, f64, "scores"), _stream(stream)))


def kvc_mi_evict(p, max_len, cache: kvc_cache, mom: kvc_moments, lse, kmax, evict_idx, evict_pos,
                 n_evict, ws, stream=None):
    i32 = torch.int32
    _check(load().kvc_mi_evict(
        ctypes.byref(p), int(max_len), ctypes.byref(cache), ctypes.byref(mom),
        _ptr(lse, torch.float32, "lse"), int(kmax), _ptr(evict_idx, i32, "evict_idx"),
        _ptr(evict_pos, i32, "evict_pos", optional=True), _ptr(n_evict, i32, "n_evict"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def kvc_zip_merge(p, new_pos, q, cache: kvc_cache, kmax, evict_idx, n_evict, partner_pos, ws,
                  stream=None):
    i32 = torch.int32
    _check(load().kvc_zip_merge(
        ctypes.byref(p), int(new_pos), _ptr(q, torch.bfloat16, "q"), ctypes.byref(cache),
        int(kmax), _ptr(evict_idx, i32, "evict_idx"), _ptr(n_evict, i32, "n_evict"),
        _ptr(partner_pos, i32, "partner_pos", optional=True), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(stream)))


def kvc_decode_step(p, t, new_pos, max_len, q, k_new, v_new, cache: kvc_cache,
                    mom: kvc_moments, o, probs, kmax, evict_idx, evict_pos, n_evict, ws,
                    stream=None):
    bf, i32 = torch.bfloat16, torch.int32
    _check(load().kvc_decode_step(
        ctypes.byref(p), int(t), int(new_pos), int(max_len), _ptr(q, bf, "q"),
        _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"), ctypes.byref(cache),
        ctypes.byref(mom), _ptr(o, torch.float32, "o"),
        _ptr(probs, torch.float64, "probs", optional=True), int(kmax),
        _ptr(evict_idx, i32, "evict_idx", optional=True),
        _ptr(evict_pos, i32, "evict_pos", optional=True), _ptr(n_evict, i32, "n_evict"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def kvc_decode_attend_noalloc(p, t, new_pos, max_len, q, k_new, v_new, cache: kvc_cache, lse,
                              f_all, probs, device_status=None, stream=None):
    """kvc_decode_attend without a workspace, for callers that cannot allocate
    device memory: the scratch is a 32 MiB static array inside the library."""
    bf = torch.bfloat16
    _check(load().kvc_decode_attend_noalloc(
        ctypes.byref(p), int(t), int(new_pos), int(max_len), _ptr(q, bf, "q"),
        _ptr(k_new, bf, "k_new"), _ptr(v_new, bf, "v_new"), ctypes.byref(cache),
        _ptr(lse, torch.float32, "lse"), _ptr(f_all, torch.float32, "f_all"),
        _ptr(probs, torch.float64, "probs", optional=True),
        _ptr(device_status, torch.int32, "device_status", optional=True), _stream(stream)))


# ------------------------------------------------------------------ prefill

def kvc_prefill_prepare(NL, Hq, Hkv, d, D, W_O, R, stream=None):
    _check(load().kvc_prefill_prepare(int(NL), int(Hq), int(Hkv), int(d), int(D),
                                      _ptr(W_O, torch.bfloat16, "W_O"),
                                      _ptr(R, torch.float32, "R"), _stream(stream)))


def kvc_prefill_workspace_size(NL, Hkv, N, B_total) -> int:
    return int(load().kvc_prefill_workspace_size(int(NL), int(Hkv), int(N), int(B_total)))


def kvc_prefill_score(NL, Hq, Hkv, d, N, w, B_total, normalize, q_win, K, V, R, scores, keep,
                      counts, idx, ws, stream=None, alloc=ALLOC_GLOBAL):
    bf = torch.bfloat16
    _check(load().kvc_prefill_score(
        int(NL), int(Hq), int(Hkv), int(d), int(N), int(w), int(B_total), int(normalize),
        int(alloc),
        _ptr(q_win, bf, "q_win"), _ptr(K, bf, "K"), _ptr(V, bf, "V"),
        _ptr(R, torch.float32, "R"), _ptr(scores, torch.float32, "scores", optional=True),
        _ptr(keep, torch.uint8, "keep"), _ptr(counts, torch.int32, "counts", optional=True),
        _ptr(idx, torch.int64, "idx", optional=True), _ptr(ws, torch.uint8, "ws", optional=True),
        0 if ws is None else ws.numel(), _stream(stream)))


def kvc_prefill_window_attention(NL, Hq, Hkv, d, N, w, row_weight, q_win, K, S, ws, stream=None):
    """row_weight: w host floats (a sequence); S: [NL][Hkv][N] fp32 output."""
    rw = (ctypes.c_float * max(1, len(row_weight)))(*[float(x) for x in row_weight])
    bf = torch.bfloat16
    _check(load().kvc_prefill_window_attention(
        int(NL), int(Hq), int(Hkv), int(d), int(N), int(w), ctypes.cast(rw, ctypes.c_void_p),
        _ptr(q_win, bf, "q_win"), _ptr(K, bf, "K"), _ptr(S, torch.float32, "S"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def kvc_prefill_snapkv(NL, Hq, Hkv, d, N, w, B_total, pool, sink, q_win, K, scores, keep, counts,
                       idx, ws, stream=None):
    bf = torch.bfloat16
    _check(load().kvc_prefill_snapkv(
        int(NL), int(Hq), int(Hkv), int(d), int(N), int(w), int(B_total), int(pool), int(sink),
        _ptr(q_win, bf, "q_win"), _ptr(K, bf, "K"),
        _ptr(scores, torch.float32, "scores", optional=True), _ptr(keep, torch.uint8, "keep"),
        _ptr(counts, torch.int32, "counts", optional=True),
        _ptr(idx, torch.int64, "idx", optional=True), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)))


def kvc_prefill_handoff_workspace_size(U, N) -> int:
    return int(load().kvc_prefill_handoff_workspace_size(int(U), int(N)))


def kvc_prefill_handoff(p, N, keep, K_src, V_src, votes_src, util_init, cache: kvc_cache,
                        mom: kvc_moments, budget, ws, stream=None):
    bf = torch.bfloat16
    _check(load().kvc_prefill_handoff(
        ctypes.byref(p), int(N), _ptr(keep, torch.uint8, "keep"), _ptr(K_src, bf, "K_src"),
        _ptr(V_src, bf, "V_src"), _ptr(votes_src, torch.int32, "votes_src", optional=True),
        _ptr(util_init, torch.float64, "util_init", optional=True), ctypes.byref(cache),
        ctypes.byref(mom), _ptr(budget, torch.int32, "budget", optional=True),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))
