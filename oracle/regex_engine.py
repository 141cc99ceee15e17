"""A small leftmost-first (Perl-style) backtracking regex matcher for the
constructs the pre-tokenizer patterns use: literals (optionally
case-insensitive), classes of one code point, greedy quantifiers over one
code point, greedy repetition of a sub-pattern, sequences, ordered
alternation and negative lookahead.

Semantics (the usual backtracking reading): an alternation tries its
branches in order; a greedy quantifier first takes as many code points as
it can and gives them back one at a time; the first way that lets the rest
of the pattern match wins.  The top-level match at position i is the first
alternative that matches at i, with the length that backtracking finds
first (not the longest).
"""

INF = float("inf")

# Simple case folding (Unicode CaseFolding.txt, status C and S) maps
# U+017F LATIN SMALL LETTER LONG S to 's' and U+212A KELVIN SIGN to 'k';
# every other code point that folds to an ASCII letter is the ASCII letter of
# the other case.
_FOLD_EXTRA = {"s": ["ſ"], "k": ["K"]}


class Node:
    pass


class Lit(Node):
    """One literal code point; icase matches every code point with the same
    simple case fold."""

    def __init__(self, ch, icase=False):
        if icase:
            lo = ch.lower()
            eq = {lo, ch.upper()} | set(_FOLD_EXTRA.get(lo, []))
            self.cps = frozenset(ord(c) for c in eq if len(c) == 1)
        else:
            self.cps = frozenset([ord(ch)])

    def one(self, cps, cls, i):
        return cps[i] in self.cps


class Cls(Node):
    """One code point whose class letter (L, N, W, O) and value satisfy a
    predicate."""

    def __init__(self, pred, name=""):
        self.pred = pred
        self.name = name

    def one(self, cps, cls, i):
        return self.pred(cps[i], cls[i])


class Seq(Node):
    def __init__(self, *items):
        self.items = items


class Alt(Node):
    def __init__(self, *branches):
        self.branches = branches


class Rep(Node):
    """Greedy quantifier {lo,hi} over a one-code-point node."""

    def __init__(self, item, lo, hi):
        assert isinstance(item, (Lit, Cls))
        self.item, self.lo, self.hi = item, lo, hi


class Star(Node):
    """Greedy repetition (X)* of a sub-pattern X of any length.  Backtracking
    order as for the recursive reading (X Star)|(empty): at each position X's
    matches are tried in X's own order, each followed by more repetitions,
    and only then the rest of the pattern.  The search keeps its own stack, so
    a long chain of repetitions needs no deep recursion."""

    def __init__(self, item):
        self.item = item


class NotAhead(Node):
    """(?!item): succeeds, consuming nothing, iff item does not match here."""

    def __init__(self, item):
        self.item = item


def _m(node, cps, cls, i, k):
    """Match node at i; on success call continuation k(j) with the end
    position j and return its result; return None if no way succeeds."""
    n = len(cps)
    if isinstance(node, (Lit, Cls)):
        if i < n and node.one(cps, cls, i):
            return k(i + 1)
        return None
    if isinstance(node, Seq):
        def run(idx, pos):
            if idx == len(node.items):
                return k(pos)
            return _m(node.items[idx], cps, cls, pos, lambda j: run(idx + 1, j))
        return run(0, i)
    if isinstance(node, Alt):
        for b in node.branches:
            r = _m(b, cps, cls, i, k)
            if r is not None:
                return r
        return None
    if isinstance(node, Rep):
        count = 0
        j = i
        while count < node.hi and j < n and node.item.one(cps, cls, j):
            count += 1
            j += 1
        while count >= node.lo:  # give back one code point at a time
            r = k(i + count)
            if r is not None:
                return r
            count -= 1
        return None
    if isinstance(node, Star):
        def ends(p):
            # every end of one match of the item at p, in backtracking order
            out = []
            _m(node.item, cps, cls, p, lambda j: out.append(j))
            return iter([j for j in out if j > p])  # an empty repetition adds nothing
        stack = [(i, ends(i))]
        while stack:
            p, it = stack[-1]
            q = next(it, None)
            if q is not None:
                stack.append((q, ends(q)))
                continue
            stack.pop()
            r = k(p)
            if r is not None:
                return r
        return None
    if isinstance(node, NotAhead):
        if _m(node.item, cps, cls, i, lambda j: j) is not None:
            return None
        return k(i)
    raise TypeError(node)


def match_at(pattern, cps, cls, i):
    """End position of the pattern's match starting at i, or None."""
    return _m(pattern, cps, cls, i, lambda j: j)
