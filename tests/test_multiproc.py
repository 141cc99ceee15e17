"""Host-side multi-rank logic on CPU (gloo, world_size 2).

The encode path shards only over independent texts: each rank encodes its
share of a batch whole, with no collective on the data path.  These tests
check the assignment (every item on exactly one rank, balanced by bytes,
identical on every rank), the reassembly in item order, and the max-over-
ranks timing reduction the benchmark uses.  Each rank encodes its items with
the oracle, which stands in for its GPU here; the gathers below exist only to
check the result.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import textgen
from exact_bpe_tokenization_utf_gb300.shard import assign_items, rank_items, reassemble
from oracle.encode import encode
from oracle.pretokenize import PATTERN_GPT2
from oracle.vocab import Vocab

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
VOCAB = os.path.join(ROOT, "data", "vocabs", "gpt2_code_1k.merges")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _items():
    rng = textgen.Rng(77)
    return [textgen.code_ascii(300 + rng.below(3000), 500 + k).encode() for k in range(9)]


def _worker(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        items = _items()
        lengths = [len(x) for x in items]
        mine = rank_items(lengths, world, rank)
        v = Vocab.load_merges(VOCAB)
        results = [encode(items[i], v, PATTERN_GPT2) for i in mine]
        # every rank derives the same assignment from the lengths alone
        got = [None] * world
        dist.all_gather_object(got, mine)
        # the benchmark's reduction: the slowest rank sets the step time
        t = torch.tensor([float(rank + 1)])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        gathered = [None] * world
        dist.all_gather_object(gathered, results)
        if rank == 0:
            out_q.put((got, gathered, float(t.item())))
    finally:
        dist.destroy_process_group()


@pytest.mark.skipif(not dist.is_available(), reason="torch.distributed unavailable")
def test_two_rank_batch_shards_and_reassembles():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got, gathered, tmax = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    items = _items()
    lengths = [len(x) for x in items]
    ref = assign_items(lengths, world)
    assert got == ref
    flat = sorted(i for a in ref for i in a)
    assert flat == list(range(len(items)))
    assert tmax == float(world)
    v = Vocab.load_merges(VOCAB)
    per_item = reassemble(gathered, ref)
    assert per_item == [encode(x, v, PATTERN_GPT2) for x in items]


def test_assignment_is_balanced_and_deterministic():
    lengths = textgen.session_batch_lengths(64, 1004)
    for world in (1, 2, 3, 4, 8):
        a = assign_items(lengths, world)
        assert a == assign_items(list(lengths), world)
        assert sorted(i for lst in a for i in lst) == list(range(len(lengths)))
        loads = [sum(lengths[i] for i in lst) for lst in a]
        # greedy longest-first: no rank exceeds the mean by more than the largest item
        assert max(loads) <= sum(lengths) / world + max(lengths)
    with pytest.raises(ValueError):
        reassemble([[1]], [[0, 1]])
