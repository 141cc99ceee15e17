"""BPE trainer for the synthetic vocabularies.

The pages train nothing; this is the usual byte-level BPE training rule,
stated here because the configurations need vocabularies with 1,000, 50,000
and 100,000 merges:

1. Pre-tokenize the corpus with the same pattern and count distinct
   fragments (as byte strings).
2. Repeat: count every adjacent symbol pair inside every fragment, weighted
   by the fragment's count (overlapping pairs such as the two (a,a) in "aaa"
   both count).  Take the pair with the largest count, ties broken by the
   smallest (left_id, right_id).  Merge it in every fragment, left to right,
   without overlap.  Its bytes get a new token id (next free id) unless a
   token with those bytes already exists, which is then reused.
3. Stop after the requested number of merges.  A pair must occur at least
   `min_count` times; if none does before the target, raise.

Byte tokens are ids 0..255 with id = byte value.  Counts are updated
incrementally, only for the fragments that contain the merged pair; the
result is the same as recounting from scratch each step (a test checks this
against `train_naive` on small corpora).
"""
import heapq
from collections import defaultdict

from .pretokenize import pretokenize
from .utf8 import decode_utf8


class TrainError(RuntimeError):
    pass


def fragment_counts(text_bytes, pattern_id):
    cps, offs = decode_utf8(text_bytes)
    counts = defaultdict(int)
    for a, b in pretokenize(cps, pattern_id):
        counts[text_bytes[offs[a]:offs[b]]] += 1
    return counts


def _merge_word(w, a, b, res):
    out = []
    i = 0
    n = len(w)
    while i < n:
        if i + 1 < n and w[i] == a and w[i + 1] == b:
            out.append(res)
            i += 2
        else:
            out.append(w[i])
            i += 1
    return out


def train_from_counts(counts, n_merges, min_count=2, progress=None):
    words = [list(k) for k in counts]
    freqs = list(counts.values())
    toks = [bytes([i]) for i in range(256)]
    index = {t: i for i, t in enumerate(toks)}
    pair_count = defaultdict(int)
    pair_words = defaultdict(set)
    for wi, w in enumerate(words):
        f = freqs[wi]
        for p in zip(w, w[1:]):
            pair_count[p] += f
            pair_words[p].add(wi)
    heap = [(-c, p[0], p[1]) for p, c in pair_count.items()]
    heapq.heapify(heap)
    merges = []
    while len(merges) < n_merges:
        while heap:
            negc, a, b = heapq.heappop(heap)
            if pair_count.get((a, b), 0) == -negc and negc < 0:
                break
        else:
            raise TrainError("no pairs left after %d merges" % len(merges))
        c = -negc
        if c < min_count:
            raise TrainError("best pair occurs %d < %d times after %d merges" % (c, min_count, len(merges)))
        tb = toks[a] + toks[b]
        res = index.get(tb)
        if res is None:
            res = len(toks)
            toks.append(tb)
            index[tb] = res
        merges.append((a, b))
        touched = set()
        for wi in pair_words.pop((a, b)):
            w = words[wi]
            f = freqs[wi]
            old = list(zip(w, w[1:]))
            if (a, b) not in old:
                continue
            nw = _merge_word(w, a, b, res)
            for p in old:
                pair_count[p] -= f
                touched.add(p)
            for p in zip(nw, nw[1:]):
                pair_count[p] += f
                pair_words[p].add(wi)
                touched.add(p)
            words[wi] = nw
        pair_count.pop((a, b), None)
        for p in touched:
            cnt = pair_count.get(p, 0)
            if cnt > 0:
                heapq.heappush(heap, (-cnt, p[0], p[1]))
            elif p in pair_count:
                del pair_count[p]
        if progress and len(merges) % progress == 0:
            print("  %d merges, last count %d" % (len(merges), c), flush=True)
    return merges


def train(text_bytes, pattern_id, n_merges, min_count=2, progress=None):
    return train_from_counts(fragment_counts(text_bytes, pattern_id), n_merges, min_count, progress)


def train_naive(counts, n_merges, min_count=1):
    """Recount every pair from scratch at every step (for tests)."""
    words = {k: list(k) for k in counts}
    toks = [bytes([i]) for i in range(256)]
    index = {t: i for i, t in enumerate(toks)}
    merges = []
    while len(merges) < n_merges:
        pc = defaultdict(int)
        for k, w in words.items():
            for p in zip(w, w[1:]):
                pc[p] += counts[k]
        if not pc:
            break
        best = min(pc.items(), key=lambda kv: (-kv[1], kv[0]))
        (a, b), c = best
        if c < min_count:
            break
        tb = toks[a] + toks[b]
        res = index.get(tb)
        if res is None:
            res = len(toks)
            toks.append(tb)
            index[tb] = res
        merges.append((a, b))
        for k in words:
            words[k] = _merge_word(words[k], a, b, res)
    return merges
