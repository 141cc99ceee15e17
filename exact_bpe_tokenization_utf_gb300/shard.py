"""Host-side sharding of independent texts over ranks (one GPU per rank).

A batch of independent texts (sessions) is the only unit the encode path
shards on: each text is encoded whole, so ranks share no data and need no
collective on the data path.  Items go to ranks greedily by byte length,
longest first (ties by item index), each to the rank with the fewest bytes so
far (ties by rank), which every rank computes identically from the lengths
alone.
"""

__all__ = ["assign_items", "rank_items", "reassemble"]


def assign_items(lengths, world):
    """Item indices per rank, each list in increasing item order."""
    if world < 1:
        raise ValueError("world must be >= 1")
    load = [0] * world
    out = [[] for _ in range(world)]
    for i in sorted(range(len(lengths)), key=lambda k: (-int(lengths[k]), k)):
        r = min(range(world), key=lambda q: (load[q], q))
        out[r].append(i)
        load[r] += int(lengths[i])
    for lst in out:
        lst.sort()
    return out


def rank_items(lengths, world, rank):
    """The item indices that `rank` encodes."""
    return assign_items(lengths, world)[rank]


def reassemble(per_rank, assignment):
    """Per-item results in item order, from each rank's results listed in
    the order of its own items."""
    n = sum(len(a) for a in assignment)
    out = [None] * n
    for items, results in zip(assignment, per_rank):
        if len(items) != len(results):
            raise ValueError("a rank returned %d results for %d items" % (len(results), len(items)))
        for i, r in zip(items, results):
            out[i] = r
    return out
