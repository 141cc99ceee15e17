"""GB300 exact byte-level BPE tokenization: Python binding of the C ABI in
include/tok.h.

This module only marshals arguments: every step of the tokenizer (UTF-8
decoding, pre-tokenization, BPE, id scatter) runs in the CUDA library
``_lib/libtokgb.so``.  Importing works without a GPU; creating a Tokenizer
needs the library (build it with ``exact_bpe_tokenization_utf_gb300._build``)
and a CUDA device, and fails loudly otherwise.

The method is the fresh-session GPU path of "TokTier: exact stateful
tokenization for agentic LLM serving" (Section 4): a GPT-style regex
pre-tokenizer recast as a run decomposition, then per-fragment BPE.
"""
from __future__ import annotations

import ctypes
import os
import struct
import zlib

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libtokgb.so")

PATTERN_GPT2 = 0
PATTERN_CL100K = 1
PATTERN_O200K = 2
PATTERN_DEEPSEEK = 3
IGNORE_MERGES = 0x100   # flag ORed into the pattern id (tok.h TOK_IGNORE_MERGES)

TOK_OK, TOK_EINVAL, TOK_EUTF8, TOK_ENOMEM, TOK_ECUDA, TOK_EBUF, TOK_ETIMEOUT, TOK_EMERGES = 0, -1, -2, -3, -4, -5, -6, -7
_NAMES = {0: "TOK_OK", -1: "TOK_EINVAL", -2: "TOK_EUTF8", -3: "TOK_ENOMEM", -4: "TOK_ECUDA", -5: "TOK_EBUF",
          -6: "TOK_ETIMEOUT", -7: "TOK_EMERGES"}

# every symbol include/tok.h declares
SYMBOLS = ["tok_load", "tok_encode", "tok_encode_offsets", "tok_repair_append", "tok_encode_batch", "tok_encode_device",
           "tok_encode_offsets_device", "tok_encode_batch_device", "tok_pretokenize", "tok_pretokenize_batch",
           "tok_last_error", "tok_error_offset", "tok_content_hash", "tok_set_timing", "tok_stage_times",
           "tok_launch_count", "tok_free", "tok_pretokenize_device_noalloc", "tok_debug_fail_alloc",
           "tok_debug_grid_wait"]


class TokError(RuntimeError):
    def __init__(self, code, msg, offset=-1):
        super().__init__("%s: %s" % (_NAMES.get(code, code), msg))
        self.code = code
        self.offset = offset


_lib = None


def lib():
    """The loaded CUDA library (ctypes).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("CUDA tokenizer library not built: %s (run exact_bpe_tokenization_utf_gb300._build)"
                          % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, U8P, U64, U32, I32P, I64P = (ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint8), ctypes.c_uint64,
                                    ctypes.c_uint32, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_int64))
    U64P = ctypes.POINTER(ctypes.c_uint64)
    L.tok_load.argtypes = [U8P, U64P, U32, ctypes.POINTER(ctypes.c_uint32), U32, ctypes.c_int,
                           ctypes.POINTER(P)]
    L.tok_encode.argtypes = [P, U8P, U64, I32P, U64, U64P]
    L.tok_encode_offsets.argtypes = [P, U8P, U64, I32P, I64P, U64, U64P]
    L.tok_repair_append.argtypes = [P, U8P, U64, U64, I32P, I64P, U64, I32P, I64P, U64, U64P, U64P]
    L.tok_encode_batch.argtypes = [P, ctypes.POINTER(U8P), U64P, U32, I32P, U64, U64P]
    L.tok_encode_device.argtypes = [P, P, U64, P, U64, P, P]
    L.tok_encode_offsets_device.argtypes = [P, P, U64, P, P, U64, P, P]
    L.tok_encode_batch_device.argtypes = [P, P, U64, P, U32, P, U64, P, P, P]
    L.tok_pretokenize.argtypes = [P, U8P, U64, I64P, U64, U64P]
    L.tok_pretokenize_batch.argtypes = [P, ctypes.POINTER(U8P), U64P, U32, I64P, U64, U64P]
    L.tok_pretokenize_device_noalloc.argtypes = [ctypes.c_int, P, U64, P, P, P]
    L.tok_pretokenize_device_noalloc.restype = ctypes.c_int
    L.tok_last_error.argtypes = [P]
    L.tok_last_error.restype = ctypes.c_char_p
    L.tok_error_offset.argtypes = [P]
    L.tok_error_offset.restype = ctypes.c_int64
    L.tok_content_hash.argtypes = [P]
    L.tok_content_hash.restype = ctypes.c_uint64
    L.tok_set_timing.argtypes = [P, ctypes.c_int]
    L.tok_stage_times.argtypes = [P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), ctypes.c_int]
    L.tok_launch_count.argtypes = [P]
    L.tok_launch_count.restype = ctypes.c_uint64
    L.tok_debug_fail_alloc.argtypes = [P, U32]
    L.tok_debug_fail_alloc.restype = ctypes.c_int
    L.tok_debug_grid_wait.argtypes = [P, U32, U32]
    L.tok_debug_grid_wait.restype = ctypes.c_int
    L.tok_free.argtypes = [P]
    L.tok_free.restype = None
    for fn in ("tok_load", "tok_encode", "tok_encode_offsets", "tok_repair_append", "tok_encode_batch", "tok_encode_device",
               "tok_encode_offsets_device", "tok_encode_batch_device", "tok_pretokenize", "tok_pretokenize_batch",
               "tok_set_timing", "tok_stage_times"):
        getattr(L, fn).restype = ctypes.c_int
    _lib = L
    return L


# --- vocabulary files ------------------------------------------------------

def read_merges_file(path):
    """Merge pairs from a zlib-compressed little-endian u32 file (magic BPEM)."""
    with open(path, "rb") as f:
        raw = zlib.decompress(f.read())
    magic, n = struct.unpack_from("<4sI", raw, 0)
    if magic != b"BPEM":
        raise ValueError("not a merges file: %s" % path)
    arr = np.frombuffer(raw, dtype="<u4", count=2 * n, offset=8)
    return arr.reshape(n, 2).astype(np.uint32)


def tokens_from_merges(merges):
    """Token byte strings implied by a merges list: ids 0..255 are the bytes,
    then each merge whose concatenated bytes are new gets the next id."""
    toks = [bytes([b]) for b in range(256)]
    seen = {t: i for i, t in enumerate(toks)}
    for a, b in np.asarray(merges).tolist():
        t = toks[a] + toks[b]
        if t not in seen:
            seen[t] = len(toks)
            toks.append(t)
    return toks


def _u8(buf):
    a = np.frombuffer(buf, dtype=np.uint8) if not isinstance(buf, np.ndarray) else buf
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


class Tokenizer:
    """One tokenizer on the current CUDA device (a tok_handle)."""

    def __init__(self, token_bytes, merges, pattern, ignore_merges=False):
        L = lib()
        self._L = L
        offs = np.zeros(len(token_bytes) + 1, dtype=np.uint64)
        offs[1:] = np.cumsum([len(t) for t in token_bytes], dtype=np.uint64)
        blob = np.frombuffer(b"".join(token_bytes), dtype=np.uint8)
        m = np.ascontiguousarray(np.asarray(merges, dtype=np.uint32).reshape(-1, 2))
        h = ctypes.c_void_p()
        rc = L.tok_load(blob.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                        offs.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), len(token_bytes),
                        m.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), m.shape[0],
                        int(pattern) | (IGNORE_MERGES if ignore_merges else 0), ctypes.byref(h))
        if rc != TOK_OK:
            raise TokError(rc, L.tok_last_error(None).decode())
        self._h = h
        self.pattern = int(pattern)
        self.ignore_merges = bool(ignore_merges)
        self.n_vocab = len(token_bytes)
        self.token_bytes = token_bytes

    @classmethod
    def from_merges(cls, merges, pattern, ignore_merges=False):
        return cls(tokens_from_merges(merges), merges, pattern, ignore_merges)

    @classmethod
    def from_merges_file(cls, path, pattern, ignore_merges=False):
        return cls.from_merges(read_merges_file(path), pattern, ignore_merges)

    def _check(self, rc):
        if rc != TOK_OK:
            raise TokError(rc, self._L.tok_last_error(self._h).decode(), self._L.tok_error_offset(self._h))

    def close(self):
        if getattr(self, "_h", None):
            self._L.tok_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- host in, host out ---------------------------------------------
    def encode(self, data):
        data = bytes(data)
        arr, p = _u8(data) if data else (None, None)
        ids = np.empty(max(len(data), 1), dtype=np.int32)
        n = ctypes.c_uint64()
        self._check(self._L.tok_encode(self._h, p, len(data), ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                       len(ids), ctypes.byref(n)))
        return ids[:n.value].copy()

    def encode_list(self, data):
        """The ids as a Python list of ints (the list output mode next to the
        id array: TokTier, Section 4.3).  The encode is the same C-ABI call
        as encode(); the list is built from its array in one conversion."""
        return self.encode(data).tolist()

    def encode_with_offsets(self, data):
        """(ids, offsets): offsets[k] is the byte offset where token k starts."""
        data = bytes(data)
        arr, p = _u8(data) if data else (None, None)
        ids = np.empty(max(len(data), 1), dtype=np.int32)
        offs = np.empty(max(len(data), 1), dtype=np.int64)
        n = ctypes.c_uint64()
        self._check(self._L.tok_encode_offsets(self._h, p, len(data),
                                               ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                               offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(ids),
                                               ctypes.byref(n)))
        return ids[:n.value].copy(), offs[:n.value].copy()

    def repair_append(self, old, old_ids, old_offsets, delta):
        """Encoding of old + delta from old's ids and token offsets (only the
        tail from the last certified cut is encoded).  Returns (ids,
        offsets, reencoded_bytes)."""
        text = bytes(old) + bytes(delta)
        arr, p = _u8(text) if text else (None, None)
        old_ids = np.ascontiguousarray(old_ids, dtype=np.int32)
        old_offsets = np.ascontiguousarray(old_offsets, dtype=np.int64)
        cap = max(len(old_ids) + len(delta) + len(old), 1)
        ids = np.empty(cap, dtype=np.int32)
        offs = np.empty(cap, dtype=np.int64)
        n, re = ctypes.c_uint64(), ctypes.c_uint64()
        self._check(self._L.tok_repair_append(
            self._h, p, len(old), len(text), old_ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            old_offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(old_ids),
            ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), offs.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            cap, ctypes.byref(n), ctypes.byref(re)))
        return ids[:n.value].copy(), offs[:n.value].copy(), re.value

    def encode_batch(self, items):
        items = [bytes(x) for x in items]
        arrs = [np.frombuffer(x, dtype=np.uint8) if x else np.zeros(1, np.uint8) for x in items]
        ptrs = (ctypes.POINTER(ctypes.c_uint8) * max(len(items), 1))(
            *[a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)) for a in arrs])
        lens = np.array([len(x) for x in items] or [0], dtype=np.uint64)
        total = int(lens[:len(items)].sum())
        ids = np.empty(max(total, 1), dtype=np.int32)
        off = np.zeros(len(items) + 1, dtype=np.uint64)
        self._check(self._L.tok_encode_batch(self._h, ptrs, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                             len(items), ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                             len(ids), off.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))))
        return ids[:int(off[-1])].copy(), off.astype(np.int64)

    def pretokenize(self, data):
        """Fragment start byte offsets (the pre-tokenizer alone)."""
        data = bytes(data)
        arr, p = _u8(data) if data else (None, None)
        starts = np.empty(max(len(data), 1), dtype=np.int64)
        n = ctypes.c_uint64()
        self._check(self._L.tok_pretokenize(self._h, p, len(data),
                                            starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(starts),
                                            ctypes.byref(n)))
        return starts[:n.value].copy()

    def pretokenize_batch(self, items):
        """Fragment starts of each item, as offsets within the item."""
        items = [bytes(x) for x in items]
        arrs = [np.frombuffer(x, dtype=np.uint8) if x else np.zeros(1, np.uint8) for x in items]
        ptrs = (ctypes.POINTER(ctypes.c_uint8) * max(len(items), 1))(
            *[a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)) for a in arrs])
        lens = np.array([len(x) for x in items] or [0], dtype=np.uint64)
        total = int(lens[:len(items)].sum())
        starts = np.empty(max(total, 1), dtype=np.int64)
        n = ctypes.c_uint64()
        self._check(self._L.tok_pretokenize_batch(self._h, ptrs, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                                  len(items), starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                                  len(starts), ctypes.byref(n)))
        flat = starts[:n.value]
        out, pos, j = [], 0, 0
        for x in items:
            k = j
            while k < len(flat) and flat[k] < pos + len(x):
                k += 1
            out.append((flat[j:k] - pos).tolist())
            j = k
            pos += len(x)
        return out

    # --- device in, device out (torch tensors or raw pointers) ---------
    def encode_device(self, d_text, n_bytes, d_ids, cap, d_status, stream=0):
        """Enqueue an encode of device bytes on `stream` (a cudaStream_t as an
        int, e.g. torch.cuda.current_stream().cuda_stream; 0 = the default
        stream); no host sync.  Pointers are ints (e.g. tensor.data_ptr());
        d_status is a device int64[4]."""
        self._check(self._L.tok_encode_device(self._h, d_text, n_bytes, d_ids, cap, d_status, stream or None))

    def encode_offsets_device(self, d_text, n_bytes, d_ids, d_offsets, cap, d_status, stream=0):
        """encode_device that also writes every token's byte offset (device
        int64, capacity cap) to d_offsets."""
        self._check(self._L.tok_encode_offsets_device(self._h, d_text, n_bytes, d_ids, d_offsets, cap, d_status,
                                                      stream or None))

    def encode_batch_device(self, d_text, n_bytes, d_item_start, n_items, d_ids, cap, d_item_off, d_status,
                            stream=0):
        self._check(self._L.tok_encode_batch_device(self._h, d_text, n_bytes, d_item_start, n_items, d_ids, cap,
                                                    d_item_off, d_status, stream or None))

    # --- introspection ---------------------------------------------------
    @property
    def content_hash(self):
        return int(self._L.tok_content_hash(self._h))

    @property
    def launch_count(self):
        return int(self._L.tok_launch_count(self._h))

    def set_timing(self, on=True):
        self._check(self._L.tok_set_timing(self._h, 1 if on else 0))

    def stage_times(self):
        ms = (ctypes.c_float * 16)()
        names = (ctypes.c_char_p * 16)()
        n = self._L.tok_stage_times(self._h, ms, names, 16)
        if n < 0:
            self._check(n)
        return {names[k].decode(): float(ms[k]) for k in range(n)}
