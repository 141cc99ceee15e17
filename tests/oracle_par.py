"""The oracle on all host cores, for the full-size parity tests.

Test infrastructure: it runs oracle.encode (unchanged) in a pool of worker
processes started with the "spawn" method, so that it is safe to create after
the GPU is in use.

A long text is cut into windows at certified cuts and the windows are
encoded independently.  A cut is a position p whose previous byte is an ASCII
letter or digit and whose own byte is ASCII but neither a letter, a digit nor
an apostrophe.  The code point before p is then a letter or a number and the
one at p has another class.  In both patterns every alternative that consumes
a letter or a number takes a maximal run of them (after at most one prefix
code point), and a contraction ends at a letter, so the match that covers
p - 1 ends at p whatever follows; no alternative looks behind, so the matches
from p on depend only on the text from p on.  This is the splice theorem of
the TokTier page (Appendix A.2) with p as the certified boundary: the encoding
of the text is the concatenation of the windows' encodings, and its fragment
starts are the windows' starts shifted by each window's offset.
tests/test_oracle_encode_trainer.py checks this against the whole-text
oracle on texts the oracle finishes in seconds.
"""
import multiprocessing as mp
import os

_VOCABS = {}

_ALNUM = frozenset(b"ABCDEFGHIJKLMNOPQRSTUVWXYZabcdefghijklmnopqrstuvwxyz0123456789")


def _vocab(path):
    v = _VOCABS.get(path)
    if v is None:
        from oracle.vocab import Vocab
        v = _VOCABS[path] = Vocab.load_merges(path) if path else Vocab.from_merges([])
    return v


def _encode_job(args):
    data, path, pattern = args
    from oracle.encode import encode_with_spans
    ids, spans = encode_with_spans(data, _vocab(path), pattern)
    return ids, [a for a, _ in spans]


def _starts_job(args):
    items, pattern = args
    from oracle.encode import pretoken_byte_spans
    return [[a for a, _ in pretoken_byte_spans(x, pattern)] for x in items]


def is_cut(data, p):
    """p is a certified cut of data (0 < p < len(data))."""
    b = data[p]
    return data[p - 1] in _ALNUM and b < 0x80 and b not in _ALNUM and b != 0x27


def windows(data, target):
    """Cut positions [0, c1, ..., len(data)]: the first certified cut at or
    after every multiple of `target` (none inside an unbroken run)."""
    n = len(data)
    out = [0]
    k = target
    while k < n:
        p = max(k, out[-1] + 1)
        while p < n and not is_cut(data, p):
            p += 1
        if p >= n:
            break
        out.append(p)
        k = p + target
    out.append(n)
    return out


class OraclePool:
    """A spawn-started pool of oracle workers; `procs` defaults to the host's
    cores."""

    def __init__(self, procs=None):
        self.procs = procs or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.procs)

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def encode_many(self, items, vocab_path, pattern):
        """[(ids, fragment starts)] of every item (largest items first)."""
        order = sorted(range(len(items)), key=lambda k: -len(items[k]))
        res = self.pool.map(_encode_job, [(items[k], vocab_path, pattern) for k in order], chunksize=1)
        out = [None] * len(items)
        for k, r in zip(order, res):
            out[k] = r
        return out

    def encode_long(self, data, vocab_path, pattern, target=1 << 17):
        """(ids, fragment starts) of one long text, window by window."""
        cuts = windows(data, target)
        parts = [data[a:b] for a, b in zip(cuts, cuts[1:])]
        res = self.encode_many(parts, vocab_path, pattern)
        ids, starts = [], []
        for a, (i, s) in zip(cuts, res):
            ids.extend(i)
            starts.extend(a + x for x in s)
        return ids, starts

    def starts_many(self, items, pattern, per_job=4000):
        """Fragment starts of every item."""
        jobs = [(items[k:k + per_job], pattern) for k in range(0, len(items), per_job)]
        out = []
        for r in self.pool.map(_starts_job, jobs, chunksize=1):
            out.extend(r)
        return out
