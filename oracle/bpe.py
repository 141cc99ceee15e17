"""Per-fragment BPE, E (TokTier, Section 4.2 and Appendix A.1: every fragment
is encoded on its own, with no state across fragments).

Rule (the textbook reading of "merges" in rank order, taken because the
pages print no listing): start from the byte tokens of the fragment; while
some adjacent pair (a, b) is in the merge table, replace the pair with the
lowest rank by its result, taking the leftmost occurrence on ties; stop
when no adjacent pair is in the table.

`mm` maps (left_id, right_id) -> (rank, result_id); a rank is the pair's
index in the merges list.

Three loops compute this; tests require them to agree:
  bpe_textbook  the rule itself, O(n^2)
  bpe_rounds    one pass per round merges every non-overlapping occurrence
                (left to right) of the minimum-rank pair.  Equal to the rule
                whenever no merge can create a pair of lower rank than its
                own, i.e. every merge that uses a token comes after every
                merge that produces it (checked by Vocab.monotone); otherwise
                not guaranteed.
  bpe_heap      a heap of (rank, position) over a linked list with lazy
                invalidation, O(n log n): equal to the rule for every merge
                table; this is what encode() uses.
"""
import heapq


def bpe_textbook(syms, mm):
    syms = list(syms)
    while True:
        best_rank, best_i, best_res = None, -1, None
        for i in range(len(syms) - 1):
            e = mm.get((syms[i], syms[i + 1]))
            if e is not None and (best_rank is None or e[0] < best_rank):
                best_rank, best_i, best_res = e[0], i, e[1]
        if best_rank is None:
            return syms
        syms[best_i:best_i + 2] = [best_res]


def bpe_rounds(syms, mm):
    syms = list(syms)
    while True:
        best = None
        for i in range(len(syms) - 1):
            e = mm.get((syms[i], syms[i + 1]))
            if e is not None and (best is None or e[0] < best[0]):
                best = (e[0], e[1], syms[i], syms[i + 1])
        if best is None:
            return syms
        _, res, a, b = best
        out = []
        i = 0
        while i < len(syms):
            if i + 1 < len(syms) and syms[i] == a and syms[i + 1] == b:
                out.append(res)
                i += 2
            else:
                out.append(syms[i])
                i += 1
        syms = out


def bpe_heap(syms, mm):
    n = len(syms)
    if n < 2:
        return list(syms)
    sym = list(syms)
    nxt = list(range(1, n + 1))
    prv = list(range(-1, n - 1))
    alive = [True] * n
    heap = []
    for i in range(n - 1):
        e = mm.get((sym[i], sym[i + 1]))
        if e is not None:
            heap.append((e[0], i, sym[i], sym[i + 1], e[1]))
    heapq.heapify(heap)
    while heap:
        rank, i, a, b, res = heapq.heappop(heap)
        j = nxt[i] if alive[i] else n
        # stale unless the pair at i is still exactly (a, b): symbols only
        # grow, so an entry can never become valid again once stale
        if j >= n or sym[i] != a or sym[j] != b:
            continue
        sym[i] = res
        alive[j] = False
        nxt[i] = nxt[j]
        if nxt[j] < n:
            prv[nxt[j]] = i
        p = prv[i]
        if p >= 0:
            e = mm.get((sym[p], sym[i]))
            if e is not None:
                heapq.heappush(heap, (e[0], p, sym[p], sym[i], e[1]))
        q = nxt[i]
        if q < n:
            e = mm.get((sym[i], sym[q]))
            if e is not None:
                heapq.heappush(heap, (e[0], i, sym[i], sym[q], e[1]))
    out = []
    i = 0
    while i < n:
        out.append(sym[i])
        i = nxt[i]
    return out
