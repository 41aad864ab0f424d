"""GPU parity of the LaProx prefill scorer (through the C ABI) against the
fp64 oracle: the full prefill-scoring workload and edge cases."""
import pytest
import torch

from kv_cache_eviction_kvc_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from parity import run_prefill_parity  # noqa: E402


def check(rep):
    print(rep)
    assert rep.ok(), rep


def test_c3_full():
    check(run_prefill_parity(W.C3))


SMALL = W.C3.with_(NL=2, N=1024, B_total=512)


@pytest.mark.parametrize("cfg,normalize", [
    (SMALL, True),
    (SMALL.with_(N=1000, B_total=777), True),            # ragged key tiles per CTA
    (SMALL.with_(N=200, w=8, B_total=1), True),          # short window, one kept
    (SMALL.with_(NL=1, Hq=8, Hkv=2, N=513, B_total=1026), True),   # keep everything
    (SMALL, False),                                       # no per-layer normalization
    (SMALL.with_(N=100, B_total=50), True),               # one CTA holds every key, 7 are empty
    (SMALL.with_(N=32, B_total=20), True),                # every key inside the window
    (SMALL.with_(NL=1, Hq=8, Hkv=2, N=40000, B_total=9000), True),   # 5000 keys per CTA
    (SMALL.with_(D_out=96), True),                        # rank-deficient Gram (rank 96 < d)
], ids=["small", "ragged", "w8-k1", "keep-all", "unnormalized", "empty-ctas", "all-window",
        "long", "rank-deficient"])
def test_prefill_edge_cases(cfg, normalize):
    check(run_prefill_parity(cfg, normalize=normalize))


@pytest.mark.parametrize("alloc", [1, 2], ids=["head-flatten", "uniform"])
def test_c3_allocations(alloc):
    check(run_prefill_parity(W.C3, alloc=alloc))


@pytest.mark.parametrize("cfg,normalize,alloc", [
    (SMALL, True, 1),
    (SMALL, True, 2),
    (SMALL.with_(N=1000, B_total=784), True, 2),          # ragged, 49 per head
    (SMALL.with_(N=1000, B_total=786), False, 1),         # unnormalized, 393 per layer
    (SMALL.with_(B_total=0), True, 2),                    # nothing kept
    (SMALL.with_(NL=1, Hq=8, Hkv=2, N=513, B_total=1026), True, 2),   # keep everything
], ids=["layer", "head", "head-ragged", "layer-unnormalized", "head-empty", "head-keep-all"])
def test_prefill_allocation_edge_cases(cfg, normalize, alloc):
    check(run_prefill_parity(cfg, normalize=normalize, alloc=alloc))


# ------------------------------------------------ window attention, SnapKV

@pytest.mark.parametrize("cfg,alpha", [
    (W.C3.with_(NL=2), 0.9),                              # full key length, KeepKV eq 15 weights
    (SMALL.with_(N=1000, w=8), 0.5),                      # ragged tiles, short window
    (SMALL.with_(N=32), 0.0),                             # every key in the window; the last query alone
], ids=["ema-c3-2layers", "ema-ragged-w8", "ema-all-window"])
def test_window_attention_ema_init(cfg, alpha):
    """KeepKV's windowed EMA initialization of the utilities on the GPU
    (weights (1 - alpha) alpha^(w-1-j) over the window rows)."""
    from parity import run_window_parity
    wts = [(1 - alpha) * alpha ** (cfg.w - 1 - j) for j in range(cfg.w)]
    err = run_window_parity(cfg, wts)
    print("max rel err", err)
    assert err <= 2e-3


@pytest.mark.parametrize("cfg,pool,sink", [
    (W.C3.with_(NL=2, B_total=2 * 8 * 128), 4, True),     # the protocol at full key length
    (SMALL.with_(N=1000, B_total=2 * 700), 4, True),      # ragged last block
    (SMALL.with_(N=200, w=8, B_total=2 * 40), 1, False),  # no pooling, no sink
    (SMALL.with_(N=513, B_total=2 * 16), 8, True),        # budget below the sinks' blocks
], ids=["snapkv-c3-2layers", "snapkv-ragged", "snapkv-plain", "snapkv-tight"])
def test_snapkv_protocol(cfg, pool, sink):
    from parity import run_snapkv_parity
    check(run_snapkv_parity(cfg, pool=pool, sink=sink))


def _sharded_worker(rank, world, port, NL, N, B):
    import os
    import torch.distributed as dist
    from kv_cache_eviction_kvc_gb300 import dist as D
    from kv_cache_eviction_kvc_gb300 import kvc as K
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        pc = W.C3.with_(NL=NL, N=N, B_total=B)
        inp = W.gen_prefill_scorer(pc, dev, 3)
        R = torch.empty(NL, pc.Hkv, pc.d, pc.d, dtype=torch.float32, device=dev)
        K.kvc_prefill_prepare(NL, pc.Hq, pc.Hkv, pc.d, pc.D, inp["W_O"], R)
        l0, l1 = D.layer_shard(NL, world, rank)
        keep_g, gflat, gs = D.prefill_score_sharded(
            l1 - l0, pc.Hq, pc.Hkv, pc.d, N, pc.w, B, inp["q_win"][l0:l1], inp["K"][l0:l1],
            inp["V"][l0:l1], R[l0:l1], l0)
        # the single-process selection over every layer
        scores = torch.empty(NL, pc.Hkv, N, dtype=torch.float32, device=dev)
        keep = torch.empty(NL, pc.Hkv, N, dtype=torch.uint8, device=dev)
        idx = torch.empty(B, dtype=torch.int64, device=dev)
        ws = torch.empty(K.kvc_prefill_workspace_size(NL, pc.Hkv, N, B), dtype=torch.uint8, device=dev)
        K.kvc_prefill_score(NL, pc.Hq, pc.Hkv, pc.d, N, pc.w, B, 1, inp["q_win"], inp["K"], inp["V"], R,
                            scores, keep, None, idx, ws)
        torch.cuda.synchronize()
        assert gflat.tolist() == idx.cpu().tolist()
        assert torch.equal(keep_g.cpu(), keep[l0:l1].cpu())
    finally:
        dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("NL,N,B", [(4, 1024, 512), (3, 640, 900)])
def test_layer_sharded_prefill_matches_single_process(NL, N, B):
    """Two ranks score a layer shard each on the GPU (the exchange over gloo;
    the ranks' kernels never wait on one another): the global selection and
    each rank's kept tokens equal the single-process kvc_prefill_score."""
    import socket
    import torch.multiprocessing as mp
    # the ranks are processes of their own on this GPU: release the memory
    # this process's allocator still caches from earlier tests
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_sharded_worker, args=(2, port, NL, N, B), nprocs=2, join=True)


def _prefill_buffers(cfg, dev):
    from kv_cache_eviction_kvc_gb300 import kvc as K
    NL, Hq, Hkv, d, N, w, B = cfg.NL, cfg.Hq, cfg.Hkv, cfg.d, cfg.N, cfg.w, cfg.B_total
    inp = W.gen_prefill_scorer(cfg, dev, 3)
    R = torch.empty(NL, Hkv, d, d, dtype=torch.float32, device=dev)
    K.kvc_prefill_prepare(NL, Hq, Hkv, d, cfg.D, inp["W_O"], R)
    ws = torch.empty(K.kvc_prefill_workspace_size(NL, Hkv, N, B), dtype=torch.uint8, device=dev)

    def outputs():
        return (torch.full((NL, Hkv, N), -1.0, dtype=torch.float32, device=dev),
                torch.full((NL, Hkv, N), 7, dtype=torch.uint8, device=dev),
                torch.full((NL, Hkv), -1, dtype=torch.int32, device=dev),
                torch.full((B,), -1, dtype=torch.int64, device=dev))

    def call(out, stream=None):
        K.kvc_prefill_score(NL, Hq, Hkv, d, N, w, B, 1, inp["q_win"], inp["K"], inp["V"], R,
                            *out, ws, stream=stream)
    return outputs, call


def _same(a, b):
    sa, ka, ca, ia = a
    sb, kb, cb, ib = b
    assert torch.equal(ka, kb) and torch.equal(ca, cb) and torch.equal(ia, ib)
    # the per-layer sums are fp64 atomics: the normalization may differ in the
    # last bit between runs
    torch.testing.assert_close(sa, sb, rtol=1e-6, atol=0.0)


def test_prefill_score_stream_order_and_graph_capture():
    """The value norms run on a library stream forked from and joined back
    into the caller's stream: results read after synchronizing only the
    caller's (non-default) stream are complete, and a CUDA graph captured
    from that stream replays the same selection."""
    dev = torch.device("cuda", 0)
    cfg = W.C3.with_(NL=4, N=4096, B_total=2048)
    outputs, call = _prefill_buffers(cfg, dev)
    ref = outputs()
    call(ref)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for _ in range(3):
        out = outputs()
        torch.cuda.current_stream().wait_stream(s)
        s.wait_stream(torch.cuda.current_stream())
        call(out, stream=s)
        s.synchronize()
        _same(ref, out)
    got = outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(got, stream=torch.cuda.current_stream())
    for _ in range(2):
        for t in got:
            t.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        _same(ref, got)
