"""The multi-process path on CPU (gloo, world size 2): the layer-sharded
prefill top-K exchange against the single-process oracle selection, and the
bench's max-over-ranks timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kv_cache_eviction_kvc_gb300 import dist as D


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = [
    # NL, Hkv, N, B_total, normalize, integer scores (ties across shards)
    (5, 2, 40, 60, True, False),
    (4, 3, 25, 90, False, True),
    (3, 1, 30, 30, True, True),
]


def _worker(rank, world, port, case):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle as O
        NL, Hkv, N, B, normalize, integer = case
        rng = np.random.default_rng(7)
        if integer:
            c = rng.integers(1, 4, size=(NL, Hkv, N)).astype(float)
            r = np.ones((NL, Hkv, N))
        else:
            c, r = rng.random((NL, Hkv, N)), rng.random((NL, Hkv, N))
        l0, l1 = D.layer_shard(NL, world, rank)
        loc = O.prefill_select(c[l0:l1], r[l0:l1], min(B, (l1 - l0) * Hkv * N),
                               normalize=normalize)
        off = l0 * Hkv * N
        flat = torch.from_numpy(loc["idx"].astype(np.int64) + off)
        scores = torch.from_numpy(loc["s"].ravel()[loc["idx"]])
        got_flat, got_s = D.gather_topk(scores, flat, B)
        ref = O.prefill_select(c, r, B, normalize=normalize)
        assert got_flat.tolist() == ref["idx"].tolist()
        np.testing.assert_array_equal(got_s.numpy(), ref["s"].ravel()[ref["idx"]])
        assert D.max_over_ranks(1.5 + rank) == 1.5 + world - 1
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", CASES, ids=["normalized", "ties-unnormalized", "one-head"])
def test_layer_sharded_topk_exchange_matches_single_process(case):
    mp.spawn(_worker, args=(2, _free_port(), case), nprocs=2, join=True)


def test_layer_shards_cover_every_layer_once():
    for NL in range(1, 12):
        for world in range(1, 5):
            got = [D.layer_shard(NL, world, r) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == NL
            assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
            sizes = [b - a for a, b in got]
            assert max(sizes) - min(sizes) <= 1


def test_merge_order_and_padding():
    s = torch.tensor([0.5, 0.7, 0.5, float("-inf"), 0.7], dtype=torch.float64)
    f = torch.tensor([9, 4, 2, D._PAD_FLAT, 1])
    flat, sc = D.merge_topk(s, f, 3)
    assert flat.tolist() == [1, 2, 4]            # 0.7 (1), 0.7 (4), then 0.5 (2 < 9)
    with pytest.raises(ValueError):
        D.merge_topk(s, f, 5)
