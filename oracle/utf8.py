"""Strict UTF-8 decoding (RFC 3629, Section 4, table of well-formed byte
sequences).

The pages do not say what the tokenizer does with malformed input; the
reading taken here is to reject it and report the byte offset where the
first malformed sequence starts, scanning left to right.  Overlong forms,
surrogates (U+D800..U+DFFF), values above U+10FFFF, truncated sequences and
stray continuation bytes are all malformed.
"""


class Utf8Error(ValueError):
    def __init__(self, offset):
        super().__init__("invalid UTF-8 at byte %d" % offset)
        self.offset = offset


# (first-byte range) -> (number of continuation bytes, allowed range of the
# second byte); every later continuation byte is 80..BF.  RFC 3629 Section 4.
_LEADS = [
    (0xC2, 0xDF, 1, 0x80, 0xBF),
    (0xE0, 0xE0, 2, 0xA0, 0xBF),
    (0xE1, 0xEC, 2, 0x80, 0xBF),
    (0xED, 0xED, 2, 0x80, 0x9F),
    (0xEE, 0xEF, 2, 0x80, 0xBF),
    (0xF0, 0xF0, 3, 0x90, 0xBF),
    (0xF1, 0xF3, 3, 0x80, 0xBF),
    (0xF4, 0xF4, 3, 0x80, 0x8F),
]


def decode_utf8(data):
    """Returns (code_points, byte_offsets) or raises Utf8Error(offset).

    byte_offsets[k] is the offset of the first byte of code point k; a final
    entry len(data) is appended."""
    cps, offs = [], []
    n = len(data)
    i = 0
    while i < n:
        b0 = data[i]
        if b0 < 0x80:
            cps.append(b0)
            offs.append(i)
            i += 1
            continue
        for lo, hi, need, s_lo, s_hi in _LEADS:
            if lo <= b0 <= hi:
                break
        else:
            raise Utf8Error(i)
        if i + need >= n:  # fewer than `need` bytes follow: truncated
            raise Utf8Error(i)
        b1 = data[i + 1]
        if not (s_lo <= b1 <= s_hi):
            raise Utf8Error(i)
        cp = b0 & (0x7F >> (need + 1))
        cp = (cp << 6) | (b1 & 0x3F)
        for k in range(2, need + 1):
            bk = data[i + k]
            if not (0x80 <= bk <= 0xBF):
                raise Utf8Error(i)
            cp = (cp << 6) | (bk & 0x3F)
        cps.append(cp)
        offs.append(i)
        i += need + 1
    offs.append(n)
    return cps, offs
