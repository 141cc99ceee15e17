"""Seeded synthetic text generators shared by the tests, the oracle's
training script and the benchmark.

This module holds no tokenizer arithmetic: it only produces strings.  All
randomness comes from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), evaluated as a counter-based
generator so that the same seed gives the same text on every machine and
every numpy version.

Workloads (sizes and mixes of the five configurations of the fresh-session
encode benchmark):

* ``code_ascii(n_bytes, seed)``      code-like ASCII (identifiers, indentation,
                                      literals, punctuation, LF lines)
* ``mixed_c2(n_bytes, seed)``         80% code ASCII, 10% CJK, 5% accented Latin,
                                      5% digit / whitespace runs (by bytes)
* ``agentic_session(n_chars, seed)``  an agent session: file dumps, tool output,
                                      JSON, shell logs, ~2% non-ASCII, some CRLF
* ``session_batch(n_items, seed)``    session lengths log-uniform in 2 KiB..1 MiB
* ``adversarial(n_bytes, seed)``      long whitespace / digit / letter runs,
                                      chained contractions, CRLF mixes, every
                                      UTF-8 length class
"""
from __future__ import annotations

import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_block(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of splitmix64 seeded with ``seed``.

    Output i is mix(seed + (i+1)*golden), the state sequence of splitmix64.
    """
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


class Rng:
    """Buffered splitmix64 stream with a few sampling helpers."""

    _BLOCK = 1 << 16

    def __init__(self, seed: int):
        self.seed = seed & 0xFFFFFFFFFFFFFFFF
        self._pos = 0
        self._buf = np.empty(0, dtype=np.uint64)
        self._i = 0

    def u64(self) -> int:
        if self._i >= len(self._buf):
            self._buf = splitmix64_block(self.seed, self._pos, self._BLOCK)
            self._buf = self._buf.tolist()
            self._pos += self._BLOCK
            self._i = 0
        v = self._buf[self._i]
        self._i += 1
        return v

    def below(self, n: int) -> int:
        """Uniform integer in [0, n) (multiply-shift, Lemire)."""
        return (self.u64() * n) >> 64

    def random(self) -> float:
        return (self.u64() >> 11) * (1.0 / 9007199254740992.0)

    def choice(self, seq):
        return seq[self.below(len(seq))]

    def geometric(self, mean: float) -> int:
        """Geometric length >= 1 with the given mean."""
        p = 1.0 / mean
        u = self.random()
        if u <= 0.0:
            u = 1e-300
        return 1 + int(math.log(u) / math.log1p(-p)) if p < 1.0 else 1

    def zipf_index(self, n: int, s: float = 1.1) -> int:
        """Index in [0, n) with probability roughly proportional to 1/(i+1)^s
        (inverse-CDF of the continuous approximation)."""
        u = self.random()
        if abs(s - 1.0) < 1e-9:
            x = math.exp(u * math.log(n + 1.0)) - 1.0
        else:
            a = 1.0 - s
            x = ((u * ((n + 1.0) ** a - 1.0)) + 1.0) ** (1.0 / a) - 1.0
        i = int(x)
        return i if i < n else n - 1


# ---------------------------------------------------------------------------
# Pools of building blocks
# ---------------------------------------------------------------------------

_SYLLABLES = [
    c + v + t
    for c in ["", "b", "c", "d", "f", "g", "h", "k", "l", "m", "n", "p", "r", "s", "t", "v", "w", "z",
              "st", "tr", "pr", "ch", "sh", "th", "gr", "cl", "fl"]
    for v in ["a", "e", "i", "o", "u", "ea", "io", "ou"]
    for t in ["", "n", "r", "s", "t", "x", "l", "m", "ck"]
]

_KEYWORDS = ["def", "return", "if", "else", "elif", "for", "while", "in", "import", "from", "class",
             "self", "None", "True", "False", "and", "or", "not", "with", "as", "try", "except",
             "raise", "yield", "lambda", "const", "let", "var", "function", "async", "await",
             "int", "void", "char", "struct", "static", "unsigned", "public", "private", "new"]

_PUNCT_OPS = [" = ", " == ", " != ", " + ", " - ", " * ", " / ", " += ", " -> ", " => ", " < ",
              " > ", " <= ", " >= ", ", ", ": ", "; ", ".", "(", ")", "[", "]", "{", "}", "::",
              " && ", " || ", " % ", " ** ", " |= ", " << ", " >> "]

_WORDS_EN = ["the", "file", "error", "value", "test", "result", "failed", "passed", "found", "line",
             "function", "expected", "got", "warning", "module", "cannot", "read", "write", "path",
             "directory", "output", "input", "running", "build", "done", "using", "version", "user",
             "request", "response", "status", "update", "created", "deleted", "changes", "commit",
             "it's", "don't", "we're", "they've", "I'm", "you'll", "she'd", "can't", "isn't", "won't"]

_ACCENTED = "àáâãäåæçèéêëìíîïðñòóôõöøùúûüýþÿÀÁÂÃÄÅÆÇÈÉÊËÌÍÎÏÐÑÒÓÔÕÖØÙÚÛÜÝĀāĂăĄąĆćČčĎďĒēĘęĚěĞğĪīİıŁłŃńŇňŌōŐőŒœŘřŚśŞşŠšŢţŤťŪūŮůŰűŸŹźŻżŽž"

_CJK_PUNCT = ["、", "。", "，", "：", "（", "）", "「", "」", "！", "？"]

_EMOJI = ["\U0001F600", "\U0001F680", "✅", "❌", "\U0001F4C1", "⚠️", "→"]


class _Pools:
    """Per-seed pools: identifiers with Zipf-like frequencies, CJK characters."""

    def __init__(self, rng: Rng, n_ident: int = 30000):
        idents = []
        seen = set()
        while len(idents) < n_ident:
            k = 1 + rng.below(3)
            parts = [rng.choice(_SYLLABLES) for _ in range(k)]
            parts = [p for p in parts if p] or ["x"]
            style = rng.below(4)
            if style == 0:
                name = "_".join(parts)
            elif style == 1:
                name = parts[0] + "".join(p.capitalize() for p in parts[1:])
            elif style == 2:
                name = "".join(p.capitalize() for p in parts)
            else:
                name = "".join(parts)
            if name and name not in seen:
                seen.add(name)
                idents.append(name)
        self.idents = idents
        # CJK characters ordered pseudo-randomly so that the Zipf head is a
        # fixed set of common characters.
        cjk = list(range(0x4E00, 0x9FFF + 1))
        for i in range(len(cjk) - 1, 0, -1):
            j = rng.below(i + 1)
            cjk[i], cjk[j] = cjk[j], cjk[i]
        self.cjk = [chr(c) for c in cjk]


def _ident(rng: Rng, pools: _Pools) -> str:
    if rng.below(10) == 0:  # fresh, rare identifier
        return "".join(rng.choice(_SYLLABLES) for _ in range(1 + rng.below(3))) or "z"
    return pools.idents[rng.zipf_index(len(pools.idents))]


def _number(rng: Rng) -> str:
    k = rng.below(6)
    if k == 0:
        return str(rng.below(10))
    if k == 1:
        return str(rng.below(1000))
    if k == 2:
        return str(rng.below(10 ** (1 + rng.below(9))))
    if k == 3:
        return "%d.%d" % (rng.below(1000), rng.below(10000))
    if k == 4:
        return "0x%x" % rng.below(1 << (4 * (1 + rng.below(8))))
    return str(rng.below(100)) + "e-" + str(rng.below(20))


def _string_lit(rng: Rng, pools: _Pools) -> str:
    words = [rng.choice(_WORDS_EN) if rng.below(2) else _ident(rng, pools) for _ in range(1 + rng.below(5))]
    q = '"' if rng.below(2) else "'"
    return q + " ".join(words) + q


def _code_line(rng: Rng, pools: _Pools) -> str:
    indent = "    " * rng.below(6)
    k = rng.below(12)
    if k == 0:
        return indent + "# " + " ".join(rng.choice(_WORDS_EN) for _ in range(2 + rng.below(8)))
    if k == 1:
        return indent + "def " + _ident(rng, pools) + "(" + ", ".join(_ident(rng, pools) for _ in range(rng.below(4))) + "):"
    if k == 2:
        return indent + "return " + _ident(rng, pools) + rng.choice(_PUNCT_OPS) + _number(rng)
    if k == 3:
        return indent + "if " + _ident(rng, pools) + rng.choice([" > ", " < ", " == ", " != "]) + _number(rng) + ":"
    if k == 4:
        return indent + _ident(rng, pools) + "." + _ident(rng, pools) + "(" + _string_lit(rng, pools) + ")"
    if k == 5:
        return indent + _ident(rng, pools) + "[" + str(rng.below(64)) + "] = " + _number(rng)
    if k == 6:
        return ""
    if k == 7:
        return indent + "for " + _ident(rng, pools) + " in range(" + _number(rng) + "):"
    if k == 8:
        return indent + rng.choice(_KEYWORDS) + " " + _ident(rng, pools) + rng.choice(_PUNCT_OPS) + _ident(rng, pools)
    if k == 9:
        return indent + "import " + _ident(rng, pools) + "." + _ident(rng, pools)
    if k == 10:
        return indent + _ident(rng, pools) + " = {" + ", ".join(
            _string_lit(rng, pools) + ": " + _number(rng) for _ in range(1 + rng.below(3))) + "}"
    parts = [_ident(rng, pools)]
    for _ in range(1 + rng.below(4)):
        parts.append(rng.choice(_PUNCT_OPS))
        parts.append(_ident(rng, pools) if rng.below(2) else _number(rng))
    return indent + "".join(parts) + rng.choice([";", "", ",", ")"])


def _cjk_run(rng: Rng, pools: _Pools) -> str:
    out = []
    for _ in range(1 + rng.below(4)):
        n = rng.geometric(6.0)
        out.append("".join(pools.cjk[rng.zipf_index(len(pools.cjk), 1.05)] for _ in range(n)))
        out.append(rng.choice(_CJK_PUNCT))
    return "".join(out)


def _accented_word(rng: Rng) -> str:
    n = 2 + rng.below(9)
    chars = []
    for _ in range(n):
        if rng.below(3) == 0:
            chars.append(_ACCENTED[rng.below(len(_ACCENTED))])
        else:
            chars.append(chr(ord("a") + rng.below(26)))
    return "".join(chars)


def _digit_ws_run(rng: Rng) -> str:
    k = rng.below(4)
    n = rng.geometric(4.0)
    if k == 0:
        return "".join(chr(ord("0") + rng.below(10)) for _ in range(n))
    if k == 1:
        return " " * n
    if k == 2:
        return "\t" * n
    return "\n" * n


def _trim_to_bytes(s: str, n_bytes: int) -> str:
    b = s.encode("utf-8")
    if len(b) >= n_bytes:
        b = b[:n_bytes]
        # step back to a code point boundary, then pad with ASCII
        while b and (b[-1] & 0xC0) == 0x80:
            b = b[:-1]
        if b and b[-1] >= 0xC0:
            b = b[:-1]
    b = b + b"x" * (n_bytes - len(b))
    return b.decode("utf-8")


def code_ascii(n_bytes: int, seed: int) -> str:
    """Code-like ASCII text of exactly ``n_bytes`` bytes."""
    rng = Rng(seed)
    pools = _Pools(rng)
    out, size = [], 0
    while size < n_bytes:
        line = _code_line(rng, pools) + "\n"
        out.append(line)
        size += len(line)
    return _trim_to_bytes("".join(out), n_bytes)


def mixed_c2(n_bytes: int, seed: int) -> str:
    """By bytes: 80% code-like ASCII, 10% CJK, 5% accented Latin, 5% runs of
    digits / spaces / tabs / newlines with geometric lengths of mean 4."""
    rng = Rng(seed)
    pools = _Pools(rng)
    out = []
    counts = [0, 0, 0, 0]
    targets = [0.80, 0.10, 0.05, 0.05]
    total = 0
    while total < n_bytes:
        # pick the component that is furthest below its target share
        k = min(range(4), key=lambda j: counts[j] - targets[j] * (total + 1))
        if k == 0:
            piece = _code_line(rng, pools) + "\n"
        elif k == 1:
            piece = _cjk_run(rng, pools)
        elif k == 2:
            piece = " ".join(_accented_word(rng) for _ in range(1 + rng.below(4))) + rng.choice([" ", ". ", ", ", "\n"])
        else:
            piece = _digit_ws_run(rng)
        nb = len(piece.encode("utf-8"))
        out.append(piece)
        counts[k] += nb
        total += nb
    return _trim_to_bytes("".join(out), n_bytes)


# --- agentic session pieces -------------------------------------------------

def _path(rng: Rng, pools: _Pools) -> str:
    return "/".join(["src"] + [_ident(rng, pools) for _ in range(1 + rng.below(3))]) + rng.choice(
        [".py", ".ts", ".rs", ".go", ".c", ".json", ".md"])


def _file_dump(rng: Rng, pools: _Pools) -> str:
    lines = []
    numbered = rng.below(2) == 0
    for i in range(5 + rng.below(60)):
        ln = _code_line(rng, pools)
        if rng.below(12) == 0:
            ln += "  # " + _cjk_run(rng, pools)
        if numbered:
            ln = "%6d\t%s" % (i + 1, ln)
        lines.append(ln)
    head = "<file path=\"" + _path(rng, pools) + "\">\n"
    return head + "\n".join(lines) + "\n</file>\n"


def _tool_output(rng: Rng, pools: _Pools) -> str:
    eol = "\r\n" if rng.below(5) == 0 else "\n"
    lines = []
    for _ in range(3 + rng.below(30)):
        k = rng.below(6)
        if k == 0:
            lines.append(_path(rng, pools) + ":" + str(1 + rng.below(2000)) + ": " + _code_line(rng, pools).strip())
        elif k == 1:
            lines.append(rng.choice(["PASSED", "FAILED", "ERROR", "SKIPPED"]) + " tests/test_" + _ident(rng, pools)
                         + ".py::" + _ident(rng, pools) + " [" + str(rng.below(101)) + "%]")
        elif k == 2:
            lines.append("error[E0" + str(100 + rng.below(900)) + "]: " + " ".join(
                rng.choice(_WORDS_EN) for _ in range(3 + rng.below(6))) + " `" + _ident(rng, pools) + "`")
        elif k == 3:
            lines.append("  --> " + _path(rng, pools) + ":" + str(rng.below(500)) + ":" + str(rng.below(80)))
        elif k == 4:
            lines.append(" ".join(rng.choice(_WORDS_EN) for _ in range(2 + rng.below(10)))
                         + (" " + rng.choice(_EMOJI) if rng.below(8) == 0 else "")
                         + (" " + _accented_word(rng) if rng.below(6) == 0 else ""))
        else:
            lines.append("=" * (10 + rng.below(60)) if rng.below(2) else "-" * (10 + rng.below(60)))
    return "<tool_output>" + eol + eol.join(lines) + eol + "</tool_output>\n"


def _json_value(rng: Rng, pools: _Pools, depth: int) -> str:
    k = rng.below(6 if depth < 3 else 4)
    if k == 0:
        return _number(rng)
    if k == 1:
        return '"' + _ident(rng, pools) + '"'
    if k == 2:
        return rng.choice(["true", "false", "null"])
    if k == 3:
        return '"' + " ".join(rng.choice(_WORDS_EN) for _ in range(1 + rng.below(6))) + '"'
    if k == 4:
        return "[" + ", ".join(_json_value(rng, pools, depth + 1) for _ in range(rng.below(5))) + "]"
    return _json_obj(rng, pools, depth + 1)


def _json_obj(rng: Rng, pools: _Pools, depth: int) -> str:
    ind = "  " * (depth + 1)
    items = ['%s"%s": %s' % (ind, _ident(rng, pools), _json_value(rng, pools, depth)) for _ in range(1 + rng.below(6))]
    return "{\n" + ",\n".join(items) + "\n" + "  " * depth + "}"


def _json_block(rng: Rng, pools: _Pools) -> str:
    return _json_obj(rng, pools, 0) + "\n"


def _shell_log(rng: Rng, pools: _Pools) -> str:
    lines = []
    for _ in range(3 + rng.below(25)):
        k = rng.below(5)
        if k == 0:
            lines.append("$ " + rng.choice(["ls -la", "git status", "make -j8", "python -m pytest -x", "cat",
                                            "grep -rn", "cd"]) + " " + _path(rng, pools))
        elif k == 1:
            lines.append("drwxr-xr-x  %d user user %6d Jan %2d %02d:%02d %s" % (
                1 + rng.below(9), rng.below(100000), 1 + rng.below(31), rng.below(24), rng.below(60),
                _ident(rng, pools)))
        elif k == 2:
            lines.append("[2026-%02d-%02d %02d:%02d:%02d.%03d] %s %s" % (
                1 + rng.below(12), 1 + rng.below(28), rng.below(24), rng.below(60), rng.below(60), rng.below(1000),
                rng.choice(["INFO", "WARN", "DEBUG", "ERROR"]),
                " ".join(rng.choice(_WORDS_EN) for _ in range(2 + rng.below(8)))))
        elif k == 3:
            p = rng.below(101)
            lines.append("[" + "=" * (p // 5) + ">" + " " * (20 - p // 5) + "] " + str(p) + "%")
        else:
            lines.append("%040x" % ((rng.u64() << 96) | (rng.u64() << 32) | rng.below(1 << 32))
                         + "  " + _path(rng, pools))
    return "\n".join(lines) + "\n"


def _session_pieces(rng: Rng, pools: _Pools):
    kinds = [(0.40, _file_dump), (0.25, _tool_output), (0.20, _json_block), (0.15, _shell_log)]
    while True:
        u = rng.random()
        acc = 0.0
        for w, f in kinds:
            acc += w
            if u < acc:
                yield f(rng, pools)
                break
        else:
            yield kinds[-1][1](rng, pools)


def agentic_session(n_chars: int, seed: int) -> str:
    """A synthetic agent session of exactly ``n_chars`` code points."""
    rng = Rng(seed)
    pools = _Pools(rng)
    out, size = [], 0
    gen = _session_pieces(rng, pools)
    while size < n_chars:
        p = next(gen)
        out.append(p)
        size += len(p)
    return "".join(out)[:n_chars]


def agentic_session_bytes(n_bytes: int, seed: int) -> str:
    """A synthetic agent session of exactly ``n_bytes`` UTF-8 bytes."""
    rng = Rng(seed)
    pools = _Pools(rng)
    out, size = [], 0
    gen = _session_pieces(rng, pools)
    while size < n_bytes:
        p = next(gen)
        out.append(p)
        size += len(p.encode("utf-8"))
    return _trim_to_bytes("".join(out), n_bytes)


def session_batch_lengths(n_items: int, seed: int, lo: int = 2048, hi: int = 1 << 20) -> list:
    """Item byte lengths, log-uniform in [lo, hi]."""
    rng = Rng(seed)
    return [int(round(math.exp(math.log(lo) + rng.random() * (math.log(hi) - math.log(lo)))))
            for _ in range(n_items)]


def session_batch(n_items: int, seed: int, lo: int = 2048, hi: int = 1 << 20) -> list:
    """A batch of fresh sessions with log-uniform byte lengths."""
    lens = session_batch_lengths(n_items, seed, lo, hi)
    return [agentic_session_bytes(n, seed * 1000 + 7 + i) for i, n in enumerate(lens)]


# --- adversarial pieces -----------------------------------------------------

_UTF8_CLASSES = ["\u0080", "߿", "ࠀ", "￿", "\U00010000", "\U0010FFFF", "\U00010400",
                 "\U0001D7D8", "\U0001F600", "²", "½", "٠", "１", "Ᲊ",
                 "é", " ", "　", " ", "\u0085", "ſ", "K"]


def adversarial_pieces(seed: int, scale: float = 1.0) -> list:
    """The adversarial components, each a separate string.

    scale < 1 shrinks the long runs proportionally (for tests that must run
    the oracle in seconds)."""
    rng = Rng(seed)
    n_ws = max(8, int(100_000 * scale))
    n_dig = max(8, int(200_000 * scale))
    n_let = max(8, int(1_000_000 * scale))
    pieces = []
    # (a) whitespace runs followed by a non-space: space only, and mixed
    pieces.append(" " * n_ws + "word")
    pieces.append("".join(rng.choice([" ", "\t", " ", "　", " "]) for _ in range(n_ws)) + "x")
    pieces.append(" " * (n_ws // 2) + "\n" + " " * (n_ws // 2) + "1")
    pieces.append("\n" * (n_ws // 2) + " " * (n_ws // 2) + ";")
    pieces.append(";" + "\r\n" * (n_ws // 4) + "  \t" + "\n" * 3 + "  y")
    # (c) long digit runs
    pieces.append("".join(chr(ord("0") + rng.below(10)) for _ in range(n_dig)) + " ")
    pieces.append("7" * (n_dig // 2 + 1) + "²٣" + "12" + ".")
    # (d) one unbroken letter run: 90% ASCII a-z, 10% 2- and 3-byte letters
    let = []
    for _ in range(n_let):
        u = rng.below(10)
        if u < 9:
            let.append(chr(ord("a") + rng.below(26)))
        elif rng.below(2):
            let.append(_ACCENTED[rng.below(len(_ACCENTED))])
        else:
            let.append(chr(0x4E00 + rng.below(0x5200)))
    pieces.append("".join(let) + " ")
    # (e) chained contractions in both cases
    conts = ["'s", "'t", "'re", "'ve", "'m", "'ll", "'d", "'S", "'T", "'RE", "'Ve", "'M", "'LL", "'lL", "'D",
             "'ſ", "'x", "''", "' s"]
    pieces.append(" ".join("".join(rng.choice(conts) for _ in range(1 + rng.below(6))) +
                           rng.choice(["", "am", "x", " ", "1", "."]) for _ in range(max(16, int(20000 * scale)))))
    # (f) mixed CRLF / LF lines
    pieces.append("".join(rng.choice(["a", "b1", " ", "\t", ";"]) + rng.choice(["\r\n", "\n", "\r", "\n\r", " \r\n "])
                          for _ in range(max(16, int(50000 * scale)))))
    # (g) every UTF-8 length class, letters / numbers / symbols / marks
    pieces.append("".join(rng.choice(_UTF8_CLASSES) + rng.choice(["", " ", "a", "1", "'", "\n"])
                          for _ in range(max(16, int(50000 * scale)))))
    # (b) a whitespace run at the very end of the text
    pieces.append("end" + " " * n_ws)
    return pieces


def adversarial(n_bytes: int, seed: int, scale: float = 1.0) -> str:
    """The adversarial components concatenated, topped up to ``n_bytes`` with
    mixed agent-session text inserted before the final whitespace run, so the
    text ends in a whitespace run that is not followed by a non-space."""
    pieces = adversarial_pieces(seed, scale)
    head = "".join(pieces[:-1])
    tail = pieces[-1]
    fill = n_bytes - len(head.encode("utf-8")) - len(tail.encode("utf-8"))
    if fill > 0:
        head += agentic_session_bytes(fill, seed + 17)
    s = head + tail
    b = s.encode("utf-8")
    if len(b) > n_bytes:
        # drop from the middle filler, never from the pinned components
        s = _trim_to_bytes(head, n_bytes - len(tail.encode("utf-8"))) + tail
    return s


def corpus(kind: str, n_bytes: int, seed: int) -> str:
    """Training corpora for the synthetic vocabularies."""
    if kind == "code":
        return code_ascii(n_bytes, seed)
    if kind == "c2":
        return mixed_c2(n_bytes, seed)
    if kind == "session":
        return agentic_session_bytes(n_bytes, seed)
    raise ValueError(kind)
