"""Pre-tokenization G: split the text into fragments with a GPT-style regex,
left to right (TokTier, Sections 3.2 and 4.1: the serial regex pass whose
every match start depends on where the previous match ended).

The pages name the tokenizer families but print no pattern.  The patterns
here are the GPT-2 pattern, the cl100k-style pattern (case-insensitive
contractions, digit groups of at most three, newline-aware whitespace), an
o200k-style pattern and a DeepSeek-style pattern, written as ASTs for
regex_engine in the same order as their regex text:

GPT-2:
  's|'t|'re|'ve|'m|'ll|'d| ?\\p{L}+| ?\\p{N}+| ?[^\\s\\p{L}\\p{N}]+|\\s+(?!\\S)|\\s+

cl100k-style:
  (?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\\r\\n\\p{L}\\p{N}]?\\p{L}+|\\p{N}{1,3}
  | ?[^\\s\\p{L}\\p{N}]+[\\r\\n]*|\\s*[\\r\\n]+|\\s+(?!\\S)|\\s+

o200k-style (this project's own definition in the style of the o200k family
the pages name: letter runs split by case, contractions as suffixes of the
word before them, and a symbol run that also takes a tail of CR, LF and '/'):
  [^\\r\\n\\p{L}\\p{N}]?[\\p{Lu}\\p{Lt}]*[\\p{Ll}\\p{Lm}\\p{Lo}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*
  |[^\\r\\n\\p{L}\\p{N}]?[\\p{Lu}\\p{Lt}]+(?:(?i:'s|'t|'re|'ve|'m|'ll|'d))*
  |\\p{N}{1,3}| ?[^\\s\\p{L}\\p{N}]+[\\r\\n/]*|\\s*[\\r\\n]+|\\s+(?!\\S)|\\s+

DeepSeek-style (this project's own definition in the style of the DeepSeek
family the pages name: the cl100k-style pattern with the letter runs of the
CJK scripts, C = letters of script extensions Han, Hiragana, Katakana or
Hangul, taken apart from other letters and without a prefix):
  (?i:'s|'t|'re|'ve|'m|'ll|'d)|[^\\r\\n\\p{L}\\p{N}]?(?:(?!C)\\p{L})+|(?:(?=C)\\p{L})+
  |\\p{N}{1,3}| ?[^\\s\\p{L}\\p{N}]+[\\r\\n]*|\\s*[\\r\\n]+|\\s+(?!\\S)|\\s+
"""
from .regex_engine import Alt, Cls, INF, Lit, NotAhead, Rep, Seq, Star, match_at
from .ucd import class_array, is_cjk, is_upper

PATTERN_GPT2 = 0
PATTERN_CL100K = 1
PATTERN_O200K = 2
PATTERN_DEEPSEEK = 3

_L = Cls(lambda cp, c: c == "L", r"\p{L}")
_N = Cls(lambda cp, c: c == "N", r"\p{N}")
_S = Cls(lambda cp, c: c == "W", r"\s")
_NOT_S = Cls(lambda cp, c: c != "W", r"\S")
_NOT_SLN = Cls(lambda cp, c: c == "O", r"[^\s\p{L}\p{N}]")
_NOT_CRLF_L_N = Cls(lambda cp, c: cp not in (10, 13) and c not in ("L", "N"), r"[^\r\n\p{L}\p{N}]")
_CRLF = Cls(lambda cp, c: cp in (10, 13), r"[\r\n]")
_SP = Lit(" ")
_UPPER = Cls(lambda cp, c: c == "L" and is_upper(cp), r"[\p{Lu}\p{Lt}]")
_LOWER = Cls(lambda cp, c: c == "L" and not is_upper(cp), r"[\p{Ll}\p{Lm}\p{Lo}]")
_CRLF_SLASH = Cls(lambda cp, c: cp in (10, 13, 47), r"[\r\n/]")
_CJK_L = Cls(lambda cp, c: c == "L" and is_cjk(cp), r"(?=C)\p{L}")
_OTHER_L = Cls(lambda cp, c: c == "L" and not is_cjk(cp), r"(?!C)\p{L}")


def _contractions(icase):
    return [Seq(*[Lit(ch, icase) for ch in "'" + tail]) for tail in ("s", "t", "re", "ve", "m", "ll", "d")]


GPT2 = Alt(
    *_contractions(False),
    Seq(Rep(_SP, 0, 1), Rep(_L, 1, INF)),
    Seq(Rep(_SP, 0, 1), Rep(_N, 1, INF)),
    Seq(Rep(_SP, 0, 1), Rep(_NOT_SLN, 1, INF)),
    Seq(Rep(_S, 1, INF), NotAhead(_NOT_S)),
    Rep(_S, 1, INF),
)

CL100K = Alt(
    Alt(*_contractions(True)),
    Seq(Rep(_NOT_CRLF_L_N, 0, 1), Rep(_L, 1, INF)),
    Rep(_N, 1, 3),
    Seq(Rep(_SP, 0, 1), Rep(_NOT_SLN, 1, INF), Rep(_CRLF, 0, INF)),
    Seq(Rep(_S, 0, INF), Rep(_CRLF, 1, INF)),
    Seq(Rep(_S, 1, INF), NotAhead(_NOT_S)),
    Rep(_S, 1, INF),
)

# the contractions after a word, any number of them (greedy)
_SUFFIX = Star(Alt(*_contractions(True)))

O200K = Alt(
    Seq(Rep(_NOT_CRLF_L_N, 0, 1), Rep(_UPPER, 0, INF), Rep(_LOWER, 1, INF), _SUFFIX),
    Seq(Rep(_NOT_CRLF_L_N, 0, 1), Rep(_UPPER, 1, INF), _SUFFIX),
    Rep(_N, 1, 3),
    Seq(Rep(_SP, 0, 1), Rep(_NOT_SLN, 1, INF), Rep(_CRLF_SLASH, 0, INF)),
    Seq(Rep(_S, 0, INF), Rep(_CRLF, 1, INF)),
    Seq(Rep(_S, 1, INF), NotAhead(_NOT_S)),
    Rep(_S, 1, INF),
)

DEEPSEEK = Alt(
    Alt(*_contractions(True)),
    Seq(Rep(_NOT_CRLF_L_N, 0, 1), Rep(_OTHER_L, 1, INF)),
    Rep(_CJK_L, 1, INF),
    Rep(_N, 1, 3),
    Seq(Rep(_SP, 0, 1), Rep(_NOT_SLN, 1, INF), Rep(_CRLF, 0, INF)),
    Seq(Rep(_S, 0, INF), Rep(_CRLF, 1, INF)),
    Seq(Rep(_S, 1, INF), NotAhead(_NOT_S)),
    Rep(_S, 1, INF),
)

PATTERNS = {PATTERN_GPT2: GPT2, PATTERN_CL100K: CL100K, PATTERN_O200K: O200K, PATTERN_DEEPSEEK: DEEPSEEK}


def pretokenize(cps, pattern_id, cls=None):
    """Fragments of a code point sequence as (start, end) code point spans.

    Matches are taken left to right: each starts where the previous one
    ended.  Every alternative consumes at least one code point and every
    class is covered, so the spans partition the text."""
    pat = PATTERNS[pattern_id]
    if cls is None:
        cls = class_array(cps)
    spans = []
    i, n = 0, len(cps)
    while i < n:
        j = match_at(pat, cps, cls, i)
        if j is None or j <= i:
            raise AssertionError("pattern failed to match at %d" % i)
        spans.append((i, j))
        i = j
    return spans
