"""Session repair after an append: the encoding of old + delta from the
encoding of old and a re-encoding of a tail (TokTier, Section 3.3 and the
splice theorem of Appendix A.2).

TEST INFRASTRUCTURE ONLY: the oracle of the library's tok_repair_append.

The cut this oracle uses follows from the patterns themselves.  Let p be a
position whose previous code point is a letter or a number and whose own code
point has another class and is not an apostrophe.  Every alternative of the
patterns that consumes a letter or a number ends at the end of a run of them
or inside it (after at most a one-code-point prefix), except that the
o200k-style pattern lets a contraction, which begins with an apostrophe,
follow a word; so the match that covers p - 1 ends exactly at p: p starts a
fragment whatever follows.  The fragments before p depend only on the text up
to and including the code point at p, and, since the patterns have no
look-behind, the fragments from p on depend only on the text from p on.  So
when the code point at p lies inside old,

    encode(old + delta) = tokens of encode(old) before p  +  encode((old + delta)[p:])

which is the splice theorem with p as the certified boundary.  The cut is the
last such p inside old; without one the whole text is encoded.
"""
import bisect

from .encode import encode_with_offsets
from .ucd import classify
from .utf8 import decode_utf8


def last_cut(old):
    """Byte offset of the last certified cut inside old (the code point at the
    cut lies in old), or 0 when old has none."""
    cps, offs = decode_utf8(old)
    cls = [classify(c) for c in cps]
    for j in range(len(cps) - 1, 0, -1):
        if cls[j - 1] in ("L", "N") and cls[j] != cls[j - 1] and cps[j] != 0x27:
            return offs[j]
    return 0


def repair_append(old, old_ids, old_offsets, delta, vocab, pattern_id):
    """(ids, offsets, reencoded_bytes) of old + delta, given old's ids and token
    byte offsets."""
    old = bytes(old)
    x = old + bytes(delta)
    p = last_cut(old)
    k = bisect.bisect_left(old_offsets, p)
    if p and (k >= len(old_offsets) or old_offsets[k] != p):
        raise ValueError("the token offsets do not belong to this text")
    ids, offs = encode_with_offsets(x[p:], vocab, pattern_id)
    return list(old_ids[:k]) + ids, list(old_offsets[:k]) + [p + o for o in offs], len(x) - p
