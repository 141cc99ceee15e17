"""Vocabularies: token byte strings plus an ordered merges list.

A merge is a pair (left_id, right_id); its rank is its index in the list.
Its result is the token whose bytes are bytes(left) + bytes(right), looked
up in the token list (so two merges that spell the same bytes share one
result).  This is the pair-keyed merges-list reading of the pages' "BPE
merges" (TokTier, Section 4.2); the pages do not say more.
"""
import hashlib
import struct
import zlib


class VocabError(ValueError):
    pass


class Vocab:
    def __init__(self, token_bytes, merges):
        self.token_bytes = [bytes(t) for t in token_bytes]
        self.merges = [(int(a), int(b)) for a, b in merges]
        index = {}
        for tid, t in enumerate(self.token_bytes):
            if t in index:
                raise VocabError("duplicate token bytes %r" % t)
            index[t] = tid
        self.index = index
        self.byte_id = []
        for b in range(256):
            tid = index.get(bytes([b]))
            if tid is None:
                raise VocabError("byte %d has no token" % b)
            self.byte_id.append(tid)
        mm = {}
        for rank, (a, b) in enumerate(self.merges):
            if not (0 <= a < len(self.token_bytes) and 0 <= b < len(self.token_bytes)):
                raise VocabError("merge %d out of range" % rank)
            if (a, b) in mm:
                raise VocabError("duplicate merge %d" % rank)
            res = index.get(self.token_bytes[a] + self.token_bytes[b])
            if res is None:
                raise VocabError("merge %d result not in vocab" % rank)
            mm[(a, b)] = (rank, res)
        self.merge_map = mm

    @classmethod
    def from_merges(cls, merges):
        """Byte tokens 0..255 (id = byte value), then one token per merge whose
        bytes are new, in merge order (the trainer's id rule)."""
        toks = [bytes([b]) for b in range(256)]
        index = {t: i for i, t in enumerate(toks)}
        for a, b in merges:
            t = toks[a] + toks[b]
            if t not in index:
                index[t] = len(toks)
                toks.append(t)
        return cls(toks, merges)

    def monotone(self):
        """True iff every merge that uses a token as an operand comes after
        every merge that produces that token (no merge can create a pair of
        lower rank than itself)."""
        last_made = {}
        for rank, (a, b) in enumerate(self.merges):
            res = self.merge_map[(a, b)][1]
            last_made[res] = rank
        first_used = {}
        for rank, (a, b) in enumerate(self.merges):
            for t in (a, b):
                first_used.setdefault(t, rank)
        return all(first_used.get(t, 1 << 62) > r for t, r in last_made.items())

    def max_token_len(self):
        return max(len(t) for t in self.token_bytes)

    def digest(self):
        h = hashlib.sha256()
        for t in self.token_bytes:
            h.update(struct.pack("<I", len(t)) + t)
        for a, b in self.merges:
            h.update(struct.pack("<II", a, b))
        return h.hexdigest()

    # --- files: zlib-compressed little-endian u32 merge pairs -----------
    def save_merges(self, path):
        raw = struct.pack("<4sI", b"BPEM", len(self.merges)) + b"".join(
            struct.pack("<II", a, b) for a, b in self.merges)
        with open(path, "wb") as f:
            f.write(zlib.compress(raw, 9))

    @classmethod
    def load_merges(cls, path):
        return cls.from_merges(read_merges(path))


def read_merges(path):
    with open(path, "rb") as f:
        raw = zlib.decompress(f.read())
    magic, n = struct.unpack_from("<4sI", raw, 0)
    if magic != b"BPEM":
        raise VocabError("bad merges file")
    vals = struct.unpack_from("<%dI" % (2 * n), raw, 8)
    return list(zip(vals[0::2], vals[1::2]))
