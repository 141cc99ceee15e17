"""encode = concatenation over fragments of BPE(fragment bytes): the two-stage
tokenizer F = E* . G (TokTier, Appendix A.1), with no normaliser, special
tokens, truncation, padding or dropout (the assumptions listed there).
decode concatenates token bytes."""
from .bpe import bpe_heap
from .pretokenize import pretokenize
from .utf8 import decode_utf8


def pretoken_byte_spans(data, pattern_id):
    """Fragments as (start_byte, end_byte) spans of the UTF-8 input."""
    cps, offs = decode_utf8(data)
    return [(offs[a], offs[b]) for a, b in pretokenize(cps, pattern_id)]


def encode_with_spans(data, vocab, pattern_id, bpe=bpe_heap, ignore_merges=False):
    """(ids, fragment byte spans): the encoding and the pre-tokenizer's
    fragments it was made from, from one pass of the pre-tokenizer.

    ignore_merges: a fragment whose bytes are a token of the vocabulary is
    that token, without BPE (TokTier, Section 4.2: the whole-word lookup of
    Llama-style tokenizers, `ignore_merges`); other fragments go through BPE
    as usual."""
    data = bytes(data)
    ids = []
    mm = vocab.merge_map
    bid = vocab.byte_id
    spans = pretoken_byte_spans(data, pattern_id)
    for a, b in spans:
        frag = data[a:b]
        if ignore_merges and frag in vocab.index:
            ids.append(vocab.index[frag])
        else:
            ids.extend(bpe([bid[x] for x in frag], mm))
    return ids, spans


def encode(data, vocab, pattern_id, bpe=bpe_heap, ignore_merges=False):
    return encode_with_spans(data, vocab, pattern_id, bpe, ignore_merges)[0]


def decode(ids, vocab):
    return b"".join(vocab.token_bytes[i] for i in ids)


def token_offsets(ids, vocab):
    """Byte offset where each token of an encoding starts: decoding
    concatenates token bytes, so token k starts where the bytes of tokens
    0..k-1 end (the byte offsets a session keeps, TokTier Sections 3.1, 3.4)."""
    out, pos = [], 0
    for i in ids:
        out.append(pos)
        pos += len(vocab.token_bytes[i])
    return out


def encode_with_offsets(data, vocab, pattern_id, bpe=bpe_heap, ignore_merges=False):
    ids = encode(data, vocab, pattern_id, bpe, ignore_merges)
    return ids, token_offsets(ids, vocab)

