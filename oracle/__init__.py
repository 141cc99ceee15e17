"""Oracle: a plain, slow, obviously correct CPU statement of exact byte-level
BPE tokenization (pre-tokenize with a GPT-style regex, then per-fragment BPE).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links anything in this package: only the tests, the smoke check and the
benchmark's CPU-baseline leg do.  It shares no code, tables or generators
with the CUDA library.

The method it states is the two-stage tokenizer F = E* . G of "TokTier:
exact stateful tokenization for agentic LLM serving" (Appendix A.1): G
splits the text into fragments (pre-tokens) with a left-to-right regex,
E encodes every fragment with BPE on its own, with no state shared across
fragments.  Sections 3.2 and 4.1 of the same page name the GPT-style
regex pre-tokenizer and its character classes; Section 4.2 names the
per-fragment BPE.  The pages print neither pattern nor a BPE listing, so
the patterns are the GPT-2 and cl100k-style patterns written out as the
configurations name them, plus an o200k-style pattern of this project's own
definition, and BPE is the textbook rule: repeatedly merge the lowest-rank
adjacent pair, leftmost first.

Modules
  utf8        strict RFC 3629 decoding with the offset of the first bad byte
  ucd         code point -> class (L, N, W, O) from committed range data
  regex_engine  a small leftmost-first backtracking matcher
  pretokenize the GPT-2 and cl100k-style patterns on that matcher
  bpe         three BPE loops (textbook, rounds, heap) that must agree
  vocab       vocabularies: token bytes, merges list, (left,right)->(rank,result)
  trainer     a BPE trainer that produces the synthetic vocabularies
  encode      encode / decode / pre-token spans in bytes

Parity pins live in tests/test_oracle_*.py.
"""
from .utf8 import Utf8Error, decode_utf8  # noqa: F401
from .ucd import classify, class_array  # noqa: F401
from .pretokenize import pretokenize, PATTERN_GPT2, PATTERN_CL100K, PATTERN_O200K, PATTERN_DEEPSEEK  # noqa: F401
from .bpe import bpe_textbook, bpe_rounds, bpe_heap  # noqa: F401
from .vocab import Vocab  # noqa: F401
from .encode import encode, decode, pretoken_byte_spans  # noqa: F401
