"""kvc_decode_attend_noalloc: the attention entry point for callers that
cannot allocate device memory (hosts that own every allocation, such as a
serving runtime with a pool reserved at start-up or a plugin interface that
passes no workspace).  Its scratch is a static array inside the library.

Checked through the C ABI against kvc_decode_attend with a workspace, on two
calls in a row over the same seeded inputs (Llama-3.1-8B attention shape,
256 units, 4096-token prefill).  This file is collected last on purpose."""
import pytest
import torch

from kv_cache_eviction_kvc_gb300 import kvc as K
from kv_cache_eviction_kvc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = 2e-3


@pytest.fixture(autouse=True)
def _free_cached_device_memory():
    """The first call on a device loads the library's device code, the
    32 MiB scratch array with it: that needs free device memory, which the
    tensors cached by earlier tests of this process may hold."""
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    yield


def _state(cfg, pre, cap, dev):
    U = cfg.U
    st = {
        "K": torch.zeros(U, cap, 128, dtype=torch.bfloat16, device=dev),
        "V": torch.zeros(U, cap, 128, dtype=torch.bfloat16, device=dev),
        "pos": torch.full((U, cap), -1, dtype=torch.int32, device=dev),
        "util": torch.full((U, cap), float("inf"), dtype=torch.float64, device=dev),
        "len": pre["len"].clone(),
    }
    st["K"][:, : cfg.N] = pre["K"][:, : cfg.N]
    st["V"][:, : cfg.N] = pre["V"][:, : cfg.N]
    st["pos"][:, : cfg.N] = pre["pos"][:, : cfg.N]
    st["cache"] = K.make_cache(st["K"], st["V"], None, st["pos"], st["util"], st["len"])
    return st


def _rel(a, b):
    return ((a - b).abs().amax(-1) / b.abs().amax(-1).clamp_min(1e-30)).max().item()


def test_noalloc_attend_matches_workspace_attend():
    dev = torch.device("cuda", 0)
    cfg = W.C1
    cap = cfg.N + 2
    pre = W.gen_prefill(cfg, dev, 0, cap=cfg.N + 1)
    ref, nal = _state(cfg, pre, cap, dev), _state(cfg, pre, cap, dev)
    p = K.make_params(cfg.U, cfg.G, cap, cfg.L, cfg.rule, cfg.alpha, cfg.T, cfg.correction)
    ws = torch.empty(K.kvc_decode_workspace_size(p), dtype=torch.uint8, device=dev)
    K.kvc_decode_workspace_init(p, ws)
    U, G = cfg.U, cfg.G
    outs = {}
    for name in ("ref", "nal"):
        outs[name] = dict(lse=torch.zeros(U, G, device=dev),
                          f_all=torch.zeros(U, G, 128, device=dev),
                          probs=torch.zeros(U, cap, dtype=torch.float64, device=dev))
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for t in (1, 2):                          # two calls in a row
        inp = W.gen_step(cfg, dev, t, 0)
        max_len = cfg.N + t
        o = outs["ref"]
        K.kvc_decode_attend(p, t, cfg.N + t - 1, max_len, inp["q"], inp["k_new"], inp["v_new"],
                            ref["cache"], o["lse"], o["f_all"], o["probs"], ws)
        o = outs["nal"]
        K.kvc_decode_attend_noalloc(p, t, cfg.N + t - 1, max_len, inp["q"], inp["k_new"],
                                    inp["v_new"], nal["cache"], o["lse"], o["f_all"], o["probs"],
                                    status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert K.kvc_get_device_status(ws) == 0
        a, b = outs["nal"], outs["ref"]
        assert (a["lse"] - b["lse"]).abs().max().item() <= TOL
        assert _rel(a["f_all"], b["f_all"]) <= TOL
        n = max_len
        pa, pb = a["probs"][:, :n], b["probs"][:, :n]
        assert ((pa - pb).abs() / pb.clamp_min(1e-300)).max().item() <= TOL
        assert torch.equal(nal["len"], ref["len"])
        assert torch.equal(nal["K"], ref["K"]) and torch.equal(nal["V"], ref["V"])
        assert torch.equal(nal["pos"], ref["pos"])


def test_noalloc_reports_device_side_shape_errors():
    """A unit whose appended length exceeds max_len is left untouched and the
    device status of the call says KVC_ERR_SHAPE (the status word lives in
    the static scratch, so it is only visible through device_status)."""
    dev = torch.device("cuda", 0)
    cfg = W.C0
    cap = cfg.N + 2
    pre = W.gen_prefill(cfg, dev, 0, cap=cfg.N + 1)
    st = _state(cfg, pre, cap, dev)
    U, G = cfg.U, cfg.G
    p = K.make_params(U, G, cap, cfg.L, cfg.rule, cfg.alpha, cfg.T, cfg.correction)
    lse = torch.zeros(U, G, device=dev)
    f_all = torch.zeros(U, G, 128, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    inp = W.gen_step(cfg, dev, 1, 0)
    len0 = st["len"].clone()
    K.kvc_decode_attend_noalloc(p, 1, cfg.N, cfg.N, inp["q"], inp["k_new"], inp["v_new"],
                                st["cache"], lse, f_all, None, status)     # max_len = len
    torch.cuda.synchronize()
    assert status.item() == 2                      # KVC_ERR_SHAPE
    assert torch.equal(st["len"], len0)
    # the next call starts from a clear status word
    K.kvc_decode_attend_noalloc(p, 1, cfg.N, cfg.N + 1, inp["q"], inp["k_new"], inp["v_new"],
                                st["cache"], lse, f_all, None, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(st["len"], len0 + 1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    dev = torch.device("cuda", 0)
    p = K.make_params(4608, 4, 32769, 3277)          # ~2.5 GB of scratch
    lse = torch.zeros(1, device=dev)
    q = torch.zeros(8, dtype=torch.bfloat16, device=dev)
    cache = K.make_cache(torch.zeros(8, dtype=torch.bfloat16, device=dev),
                         torch.zeros(8, dtype=torch.bfloat16, device=dev), None,
                         torch.zeros(1, dtype=torch.int32, device=dev),
                         torch.zeros(1, dtype=torch.float64, device=dev),
                         torch.zeros(1, dtype=torch.int32, device=dev))
    with pytest.raises(K.KvcError) as ei:
        K.kvc_decode_attend_noalloc(p, 1, 0, 10, q, q, q, cache, lse, lse, None)
    assert ei.value.status == 6 and "static scratch" in str(ei.value)
