"""Multi-process plumbing for running the path on several GPUs of one node
(one process per GPU, torch.distributed).  No arithmetic of the method
happens here beyond ordering the candidates of the one exchange.

* Decode units (sequence, layer, KV head) are independent: each rank runs its
  own units and the only collective is the bench's max over ranks of the
  timed region.
* The LaProx prefill scorer shards by layer, so the per-layer normalization
  stays inside a rank; the global top-K (LaProx key design 3) then needs one
  exchange.  Every element of the global top-B_total is also in its own
  shard's top-B_total (fewer than B_total elements outrank it overall, so
  fewer than B_total do inside its shard), so each rank contributes its
  local top-B_total (score, flat index) pairs, and the merge of the gathered
  pairs in the selection's order (score descending, flat index ascending) is
  exactly the single-process selection.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

_PAD_FLAT = torch.iinfo(torch.int64).max


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over the ranks of the default group (the bench's
    timed region is the slowest rank's)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def layer_shard(NL: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous layer range [l0, l1) of `rank`; the first NL % world ranks
    take one layer more."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank outside the world")
    base, extra = divmod(NL, world)
    l0 = rank * base + min(rank, extra)
    return l0, l0 + base + (1 if rank < extra else 0)


def merge_topk(scores: torch.Tensor, flat: torch.Tensor, B_total: int):
    """The B_total best (score, flat) pairs in the selection's order (score
    descending, then flat index ascending), returned as (flat ascending,
    their scores).  Padding pairs carry flat = int64 max and sort last."""
    order = torch.argsort(flat, stable=True)
    s1, f1 = scores[order], flat[order]
    order = torch.argsort(-s1, stable=True)          # ties keep ascending flat
    s2, f2 = s1[order][:B_total], f1[order][:B_total]
    if (f2 == _PAD_FLAT).any():
        raise ValueError("fewer candidates than B_total")
    back = torch.argsort(f2)
    return f2[back], s2[back]


def gather_topk(scores: torch.Tensor, flat: torch.Tensor, B_total: int, group=None):
    """One exchange of the layer-sharded prefill scorer: this rank's local
    top-B_total pairs (scores fp32/fp64, flat int64 global indices, at most
    B_total of them) are all-gathered and merged.  Returns the global
    (flat ascending, scores) on every rank."""
    n = int(flat.numel())
    if n > B_total:
        raise ValueError("a rank may contribute at most B_total pairs")
    dev = scores.device
    s = torch.full((B_total,), float("-inf"), dtype=torch.float64, device=dev)
    f = torch.full((B_total,), _PAD_FLAT, dtype=torch.int64, device=dev)
    s[:n] = scores.to(torch.float64)
    f[:n] = flat.to(torch.int64)
    world = dist.get_world_size(group)
    ss = [torch.empty_like(s) for _ in range(world)]
    fs = [torch.empty_like(f) for _ in range(world)]
    dist.all_gather(ss, s, group=group)
    dist.all_gather(fs, f, group=group)
    return merge_topk(torch.cat(ss), torch.cat(fs), B_total)


def prefill_score_sharded(NL_local: int, Hq: int, Hkv: int, d: int, N: int, w: int, B_total: int,
                          q_win, K, V, R, l0: int, normalize: int = 1, group=None, stream=None):
    """The layer-sharded LaProx scorer: this rank's layers [l0, l0 + NL_local)
    (q_win [NL_local][Hq][w][d], K, V [NL_local][Hkv][N][d], R [NL_local]
    [Hkv][d][d], on this rank's GPU) are scored by kvc_prefill_score with the
    rank's own per-layer normalization and its local top-min(B_total, shard)
    selection; one exchange (gather_topk: on the device over NCCL, through the
    host over gloo) gives the global top-B_total.  Returns (keep
    [NL_local][Hkv][N] uint8 under the global selection, the global flat
    indices ascending, their scores)."""
    from . import kvc as K_
    dev = K.device
    n_local = NL_local * Hkv * N
    b_local = min(int(B_total), n_local)
    scores = torch.empty(NL_local, Hkv, N, dtype=torch.float32, device=dev)
    keep = torch.empty(NL_local, Hkv, N, dtype=torch.uint8, device=dev)
    idx = torch.empty(b_local, dtype=torch.int64, device=dev)
    ws = torch.empty(K_.kvc_prefill_workspace_size(NL_local, Hkv, N, b_local), dtype=torch.uint8,
                     device=dev)
    K_.kvc_prefill_score(NL_local, Hq, Hkv, d, N, w, b_local, normalize, q_win, K, V, R, scores,
                         keep, None, idx, ws, stream)
    off = l0 * Hkv * N
    xdev = dev if dist.get_backend(group) == "nccl" else torch.device("cpu")
    gflat, gs = gather_topk(scores.view(-1)[idx].to(xdev), (idx + off).to(xdev), int(B_total), group)
    mine = gflat[(gflat >= off) & (gflat < off + n_local)] - off
    keep_g = torch.zeros(n_local, dtype=torch.uint8, device=dev)
    keep_g[mine.to(dev)] = 1
    return keep_g.view(NL_local, Hkv, N), gflat, gs
