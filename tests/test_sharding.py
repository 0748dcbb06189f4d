"""The multi-GPU path on CPU: text partitioning and the result gather over
world-size-2 `gloo` process groups (no GPU involved).

Each rank stands in for one GPU: it encodes its texts with a per-text
function that depends on the text alone (a deterministic unit vector from the
text's ids, or the CPU oracle's encoder on the tiny shape), exactly the
property that makes the encoder shard by text.  The gathered result must
equal the single-process result in input order.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from text_embedding_encoder_gb300 import sharding, synth


def _per_text_vector(ids, width=16):
    rng = np.random.default_rng(int(np.sum(ids.astype(np.int64) * np.arange(1, len(ids) + 1))) % (2 ** 32))
    v = rng.standard_normal(width)
    return (v / np.linalg.norm(v)).astype(np.float32)


def _encode_all(ids, cu, width=16):
    rows = [_per_text_vector(ids[cu[j]:cu[j + 1]], width) for j in range(len(cu) - 1)]
    return np.stack(rows) if rows else np.zeros((0, width), np.float32)


def test_partition_covers_every_text_once_and_balances():
    ids, cu = synth.sweep_batch(8192, 3, 1000)
    for world in (1, 2, 3, 8):
        parts = sharding.partition_texts(cu, world)
        allt = np.sort(np.concatenate(parts))
        np.testing.assert_array_equal(allt, np.arange(len(cu) - 1))
        loads = [int(np.diff(cu)[p].sum()) for p in parts]
        assert max(loads) - min(loads) <= int(np.diff(cu).max())   # greedy bound: one text
    assert sharding.partition_texts(cu, 2)[0].tolist() == sharding.partition_texts(cu, 2)[0].tolist()


def test_shard_batch_keeps_each_text_intact():
    ids, cu = synth.make_batch([5, 1, 9, 3], 100, seed=1)
    sub_ids, sub_cu = sharding.shard_batch(ids, cu, [2, 0])
    np.testing.assert_array_equal(sub_cu, [0, 9, 14])
    np.testing.assert_array_equal(sub_ids[:9], ids[6:15])
    np.testing.assert_array_equal(sub_ids[9:], ids[0:5])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ids, cu, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        texts = sharding.partition_texts(cu, world)[rank]
        sub_ids, sub_cu = sharding.shard_batch(ids, cu, texts)
        local = _encode_all(sub_ids, sub_cu)
        full = sharding.gather_embeddings(local, texts, len(cu) - 1, width=16)
        q.put((rank, full))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lengths", [[37, 150, 8, 64, 129, 3], [500], [2, 2]])   # [500]: one rank gets no text
def test_two_rank_gather_matches_single_process(lengths):
    ids, cu = synth.make_batch(lengths, 4096, seed=len(lengths))
    want = _encode_all(ids, cu)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ids, cu, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        np.testing.assert_array_equal(results[r], want)


def _oracle_worker(rank, world, port, ids, cu, q):
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        model = oracle.OracleModel(synth.make_weights(synth.TINY, seed=0), synth.TINY, "fp32")
        calls = []

        def encode_fn(sub_ids, sub_cu):
            calls.append(len(sub_cu) - 1)
            return oracle.encode_packed(sub_ids, sub_cu, model)

        full = sharding.encode_sharded(encode_fn, ids, cu, synth.TINY.hidden)
        q.put((rank, full, calls))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lengths", [[37, 150, 8, 64, 129, 3], [60]])   # [60]: rank 1 encodes nothing
def test_encode_sharded_with_the_oracle_as_encoder(lengths):
    """encode_sharded, the multi-GPU helper the library's Encoder.encode plugs
    into, run over two gloo ranks with the oracle as each rank's encoder: the
    gathered vectors equal the oracle's single-process encoding of the batch."""
    import oracle
    ids, cu = synth.make_batch(lengths, synth.TINY.vocab, seed=3)
    model = oracle.OracleModel(synth.make_weights(synth.TINY, seed=0), synth.TINY, "fp32")
    want = oracle.encode_packed(ids, cu, model).astype(np.float32)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_oracle_worker, args=(r, 2, port, ids, cu, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(2):
        r, full, calls = q.get(timeout=300)
        results[r] = (full, calls)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        np.testing.assert_array_equal(results[r][0], want)
    assert sum(sum(c) for _, c in results.values()) == len(lengths)   # every text encoded exactly once
    if len(lengths) == 1:
        assert results[1][1] == []
