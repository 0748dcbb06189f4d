"""Data-parallel sharding of a packed batch over several GPUs (one process per GPU).

Texts are independent (positions restart per text and attention never leaves
a text), so a batch shards by whole texts with replicated weights and no
exchange during the pass.  The host assigns texts to ranks (largest first to
the least-loaded rank, so token counts balance), each rank encodes its
sub-batch on its own GPU, and the unit vectors come back to their input order
with one all-gather of the per-rank results after the pass.
"""
from __future__ import annotations

import heapq

import numpy as np


def partition_texts(cu_seqlens, world: int) -> list:
    """Assign every text to one of `world` ranks, balancing token counts.

    Returns one sorted int64 array of text indices per rank.  Deterministic:
    texts are taken longest first (ties by index) and each goes to the rank
    with the fewest tokens so far (ties by rank).
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    order = sorted(range(len(lens)), key=lambda j: (-int(lens[j]), j))
    heap = [(0, r) for r in range(world)]
    parts = [[] for _ in range(world)]
    for j in order:
        load, r = heapq.heappop(heap)
        parts[r].append(j)
        heapq.heappush(heap, (load + int(lens[j]), r))
    return [np.array(sorted(p), dtype=np.int64) for p in parts]


def shard_batch(ids, cu_seqlens, texts):
    """The sub-batch of the given text indices: (ids int32[T_r], cu int32[n_r + 1])."""
    ids = np.asarray(ids)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    pieces = [ids[cu[j]:cu[j + 1]] for j in texts]
    sub_ids = np.concatenate(pieces).astype(np.int32) if pieces else np.zeros(0, np.int32)
    sub_cu = np.zeros(len(texts) + 1, dtype=np.int32)
    sub_cu[1:] = np.cumsum([cu[j + 1] - cu[j] for j in texts])
    return sub_ids, sub_cu


def gather_embeddings(local_out, texts, n_texts: int, width: int, group=None):
    """All-gather each rank's [n_r, width] unit vectors into the [n_texts, width] result in input order.

    `local_out` is a host array (or CPU tensor) of this rank's vectors, row i
    belonging to text `texts[i]`; a rank with no texts passes an empty array.
    Uses torch.distributed with the default (or given) process group; every
    rank returns the full result.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    local = torch.as_tensor(np.ascontiguousarray(local_out, dtype=np.float32).reshape(-1, width))
    idx = torch.as_tensor(np.asarray(texts, dtype=np.int64))
    counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(counts, torch.tensor([idx.numel()], dtype=torch.int64), group=group)
    max_n = max(1, int(max(c.item() for c in counts)))
    pad_out = torch.zeros(max_n, width, dtype=torch.float32)
    pad_idx = torch.full((max_n,), -1, dtype=torch.int64)
    pad_out[: idx.numel()] = local
    pad_idx[: idx.numel()] = idx
    outs = [torch.empty_like(pad_out) for _ in range(world)]
    idxs = [torch.empty_like(pad_idx) for _ in range(world)]
    dist.all_gather(outs, pad_out, group=group)
    dist.all_gather(idxs, pad_idx, group=group)
    result = np.full((n_texts, width), np.nan, dtype=np.float32)
    for o, i in zip(outs, idxs):
        keep = i >= 0
        result[i[keep].numpy()] = o[keep].numpy()
    return result


def encode_sharded(encode_fn, ids, cu_seqlens, width: int, group=None):
    """Encode a packed batch over all ranks of a process group, one GPU per rank.

    Every rank calls this with the same host batch (ids int32[T], cu_seqlens
    int32[n + 1]).  The texts are partitioned by `partition_texts`, this rank
    encodes its own sub-batch with `encode_fn(sub_ids, sub_cu) -> [n_r, width]`
    (one row per text: for the library, ``Encoder.encode`` of a context on this
    rank's GPU), and the vectors are all-gathered back into input order.  A rank that
    receives no text does not call `encode_fn`.  Every rank returns the full
    [n, width] float32 result.  There is no exchange during the pass itself:
    texts are independent (positions restart per text and attention stays
    inside it).
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = cu.shape[0] - 1
    texts = partition_texts(cu, world)[rank]
    if len(texts):
        sub_ids, sub_cu = shard_batch(ids, cu, texts)
        local = np.asarray(encode_fn(sub_ids, sub_cu), dtype=np.float32).reshape(len(texts), width)
    else:
        local = np.zeros((0, width), dtype=np.float32)
    return gather_embeddings(local, texts, n, width, group=group)
