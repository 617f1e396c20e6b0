"""CPU oracle for byte-level BPE encoding (ctypes wrapper over bpe_oracle.c).

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import this package. The product path (the
byte_level_bpe_gb300 package and its CUDA library) never imports it, and this
package never imports the product.

The oracle is a plain single-threaded C implementation written from the pages:
"tiktoken Deep Dive" (split pattern, parts-vector merge loop, specials, byte
floor, decode) and "Making Kimi K3 Tokenization 18x Faster For Million Token
Agentic Workloads" (typed segments, safe chunking). Every function in the C
file names the section it follows.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bpe_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

ORC_OK = 0
ORC_E_CAPACITY = -4
ORC_E_UTF8 = -3
ORC_E_BADID = -8

_lib = None


def build(force=False):
    """Compiles the oracle with gcc (plain C99, -O2) into oracle/_build."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    deps = [SRC, os.path.join(HERE, "unicode_ranges.h")]
    if not force and os.path.exists(LIB_PATH):
        if os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(d) for d in deps):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-Wall", "-shared", "-fPIC",
                           SRC, "-o", tmp])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        _lib.orc_new.argtypes = [P, P, P, I64, P, P, P, I64, ctypes.POINTER(P)]
        _lib.orc_new.restype = ctypes.c_int
        _lib.orc_free.argtypes = [P]
        _lib.orc_encode_segments.argtypes = [P, P, P, P, I64, ctypes.c_int, P, I64, P,
                                             ctypes.POINTER(I64), ctypes.POINTER(I64)]
        _lib.orc_encode_segments.restype = ctypes.c_int
        _lib.orc_decode.argtypes = [P, P, I64, P, I64, ctypes.POINTER(I64)]
        _lib.orc_decode.restype = ctypes.c_int
        _lib.orc_bpe_piece.argtypes = [P, P, I64, P]
        _lib.orc_bpe_piece.restype = I64
        _lib.orc_split_bytes.argtypes = [P, I64, P, ctypes.c_int]
        _lib.orc_split_bytes.restype = I64
        _lib.orc_safe_chunks_bytes.argtypes = [P, I64, P]
        _lib.orc_safe_chunks_bytes.restype = I64
        _lib.orc_cp_class.argtypes = [ctypes.c_uint32]
        _lib.orc_cp_class.restype = ctypes.c_int
        _lib.orc_py_isspace.argtypes = [ctypes.c_uint32]
        _lib.orc_py_isspace.restype = ctypes.c_int
        _lib.orc_train.argtypes = [P, I64, I64, P, I64, P]
        _lib.orc_train.restype = I64
        _lib.orc_utf8_holdback.argtypes = [P, I64]
        _lib.orc_utf8_holdback.restype = ctypes.c_int
        _lib.orc_set_pattern.argtypes = [P, ctypes.c_int]
        _lib.orc_set_pattern.restype = ctypes.c_int
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


def _buf(b):
    """bytes -> uint8 array (keeps a reference alive with the caller)."""
    return np.frombuffer(b, dtype=np.uint8) if len(b) else np.zeros(1, np.uint8)


class OracleError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"oracle error {code}: {msg}")
        self.code = code


class Encoding:
    """ranks: list of byte strings where index = rank = id (or (bytes, id) pairs);
    specials: dict str|bytes -> id."""

    def __init__(self, ranks, specials=None, pattern=None):
        if ranks and isinstance(ranks[0], tuple):
            toks = [t for t, _ in ranks]
            ids = [i for _, i in ranks]
        else:
            toks = list(ranks)
            ids = list(range(len(toks)))
        self.n = len(toks)
        self._rank_bytes = _buf(b"".join(toks))
        self._rank_off = np.zeros(len(toks) + 1, np.int64)
        np.cumsum([len(t) for t in toks], out=self._rank_off[1:])
        self._rank_ids = np.asarray(ids, np.uint32)
        specials = specials or {}
        sb = [s.encode() if isinstance(s, str) else s for s in specials]
        self._spec_bytes = _buf(b"".join(sb))
        self._spec_off = np.zeros(len(sb) + 1, np.int64)
        if sb:
            np.cumsum([len(s) for s in sb], out=self._spec_off[1:])
        self._spec_ids = np.asarray(list(specials.values()), np.int32)
        h = ctypes.c_void_p()
        rc = lib().orc_new(_ptr(self._rank_bytes), _ptr(self._rank_off), _ptr(self._rank_ids),
                           self.n, _ptr(self._spec_bytes), _ptr(self._spec_off),
                           _ptr(self._spec_ids), len(sb), ctypes.byref(h))
        if rc != ORC_OK:
            raise OracleError(rc, "table rejected")
        self._h = h
        if pattern is not None:
            rc = lib().orc_set_pattern(h, int(pattern))
            if rc != ORC_OK:
                raise OracleError(rc, "unknown pattern")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.orc_free(h)
            self._h = None

    def encode_segments(self, segments, tiktoken_safe=False):
        """segments: list of (bytes|str, allow_special) -> (ids int32 array, offsets int64)."""
        parts = [s.encode("utf-8", "surrogatepass") if isinstance(s, str) else s
                 for s, _ in segments]
        text = b"".join(parts)
        seg_off = np.zeros(len(parts) + 1, np.int64)
        if parts:
            np.cumsum([len(p) for p in parts], out=seg_off[1:])
        allow = np.asarray([1 if a else 0 for _, a in segments] or [0], np.uint8)
        return self.encode_arrays(_buf(text), seg_off, allow, len(parts), tiktoken_safe)

    def encode_arrays(self, text_u8, seg_off, allow_u8, S, tiktoken_safe=False):
        text_u8 = np.ascontiguousarray(text_u8, np.uint8)
        seg_off = np.ascontiguousarray(seg_off, np.int64)
        allow_u8 = np.ascontiguousarray(allow_u8, np.uint8)
        cap = max(int(seg_off[S]) if S else 0, 1)
        out = np.zeros(cap, np.int32)
        offs = np.zeros(S + 1, np.int64)
        n = ctypes.c_int64(0)
        bad = ctypes.c_int64(-1)
        rc = lib().orc_encode_segments(self._h, _ptr(text_u8), _ptr(seg_off), _ptr(allow_u8),
                                       S, 1 if tiktoken_safe else 0, _ptr(out), cap,
                                       _ptr(offs), ctypes.byref(n), ctypes.byref(bad))
        if rc != ORC_OK:
            raise OracleError(rc, f"encode failed (bad byte at {bad.value})")
        return out[: n.value].copy(), offs

    def encode(self, text, allow_special=False, tiktoken_safe=False):
        ids, _ = self.encode_segments([(text, allow_special)], tiktoken_safe)
        return ids

    def bpe_piece(self, piece):
        b = _buf(piece)
        out = np.zeros(max(len(piece), 1), np.int32)
        k = lib().orc_bpe_piece(self._h, _ptr(b), len(piece), _ptr(out))
        if k < 0:
            raise OracleError(int(k), "bpe failed")
        return out[:k].copy()

    def decode(self, ids):
        ids = np.ascontiguousarray(ids, np.int32)
        n = ctypes.c_int64(0)
        lib().orc_decode(self._h, _ptr(ids), len(ids), None, 0, ctypes.byref(n))
        out = np.zeros(max(n.value, 1), np.uint8)
        rc = lib().orc_decode(self._h, _ptr(ids), len(ids), _ptr(out), n.value, ctypes.byref(n))
        if rc != ORC_OK:
            raise OracleError(rc, "decode failed")
        return out[: n.value].tobytes()


def utf8_holdback(b):
    """How many trailing bytes of b form a proper prefix of a UTF-8 character."""
    arr = _buf(bytes(b))
    return int(lib().orc_utf8_holdback(_ptr(arr), len(arr)))


class StreamDecoder:
    """Streaming decode ("tiktoken Deep Dive", "Pitfalls that bite in
    production"): each feed returns the held-back bytes of the previous feed
    plus the bytes of the new ids, minus a trailing partial character, which
    waits for the next feed; finish() returns what is still held."""

    def __init__(self, enc):
        self.enc = enc
        self.pending = b""

    def feed(self, ids):
        out = self.pending + self.enc.decode(ids)
        k = utf8_holdback(out)
        self.pending = out[len(out) - k:] if k else b""
        return out[:len(out) - k]

    def finish(self):
        out, self.pending = self.pending, b""
        return out


PATTERN_CL100K = 1       # the split pattern printed on the tiktoken page
PATTERN_R50K_DIGITS = 2  # the same with r50k's digit clause " ?\p{N}++"


def split(text, pattern=PATTERN_CL100K):
    """Pre-token byte strings of one ordinary piece (the pattern's clauses)."""
    b = text.encode("utf-8", "surrogatepass") if isinstance(text, str) else text
    arr = _buf(b)
    st = np.zeros(len(b) + 1, np.int64)
    k = lib().orc_split_bytes(_ptr(arr), len(b), _ptr(st), int(pattern))
    if k < 0:
        raise OracleError(int(k), "split failed")
    starts = list(st[:k]) + [len(b)]
    return [b[starts[i]:starts[i + 1]] for i in range(k)]


def safe_chunks(text):
    """Byte strings of the tiktoken-safe chunks of one segment."""
    b = text.encode("utf-8", "surrogatepass") if isinstance(text, str) else text
    arr = _buf(b)
    st = np.zeros(len(b) + 1, np.int64)
    k = lib().orc_safe_chunks_bytes(_ptr(arr), len(b), _ptr(st))
    if k < 0:
        raise OracleError(int(k), "chunking failed")
    starts = list(st[:k]) + [len(b)]
    return [b[starts[i]:starts[i + 1]] for i in range(k)]


def cp_class(c):
    """0 = other, 1 = \\p{L}, 2 = \\p{N}, 3 = \\s."""
    return lib().orc_cp_class(c)


def py_isspace(c):
    return bool(lib().orc_py_isspace(c))


def train(corpus, n_merges):
    """The plain BPE trainer: returns the learned token byte strings (ranks 256..)."""
    arr = _buf(corpus)
    cap = 64 * n_merges + 1024
    toks = np.zeros(cap, np.uint8)
    off = np.zeros(n_merges + 1, np.int64)
    k = lib().orc_train(_ptr(arr), len(corpus), n_merges, _ptr(toks), cap, _ptr(off))
    if k < 0:
        raise OracleError(int(k), "training failed")
    return [toks[off[i]:off[i + 1]].tobytes() for i in range(k)]
