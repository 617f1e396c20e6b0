"""Thin ctypes binding of libtk (include/tk.h): argument marshalling only.

Every step of encoding runs in libtk's CUDA kernels. The functions here keep
the C ABI's names and argument order; torch is used only to own device
memory and to name the current CUDA stream. If the library is missing or no
GPU is present the calls raise: there is no CPU fallback.
"""
import ctypes
import os

from . import build as _build

TK_OK = 0
TK_E_ARG = -1
TK_E_TABLE = -2
TK_E_UTF8 = -3
TK_E_CAPACITY = -4
TK_E_CUDA = -5
TK_E_NOMEM = -6
TK_E_TIMEOUT = -7
TK_E_BADID = -8
TK_E_LIMIT = -9
TK_PATTERN_CL100K = 1
TK_PATTERN_R50K_DIGITS = 2

# Every exported function of include/tk.h, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
SIGNATURES = {
    "tk_load": (_INT, [_P, _P, _P, _I64, _P, _P, _P, _I64, _INT, ctypes.POINTER(_P)]),
    "tk_free": (None, [_P]),
    "tk_workspace_create": (_INT, [_P, _I64, _I64, ctypes.POINTER(_P)]),
    "tk_workspace_free": (None, [_P]),
    "tk_encode_segments": (_INT, [_P, _P, _P, _I64, _P, _P, _I64, _INT, _P, _I64, _P,
                                  ctypes.POINTER(_I64), _P]),
    "tk_encode_segments_host": (_INT, [_P, _P, _P, _I64, _P, _P, _I64, _INT, _P, _I64, _P,
                                       ctypes.POINTER(_I64), _P]),
    "tk_decode": (_INT, [_P, _P, _P, _I64, _P, _I64, ctypes.POINTER(_I64), _P]),
    "tk_decode_noalloc": (_INT, [_P, _P, _I64, _P, _I64, ctypes.POINTER(_I64), _P]),
    "tk_decode_stream": (_INT, [_P, _P, _P, _P, _I64, _INT, _P, _I64, ctypes.POINTER(_I64), _P]),
    "tk_decode_segments": (_INT, [_P, _P, _P, _I64, _P, _I64, _P, _I64, _P, ctypes.POINTER(_I64), _P]),
    "tk_n_ranks": (_I64, [_P]),
    "tk_n_specials": (_I64, [_P]),
    "tk_max_id": (_I64, [_P]),
    "tk_profile_enable": (_INT, [_P, _INT]),
    "tk_profile_read": (_INT, [_P, _INT, ctypes.POINTER(ctypes.c_char_p),
                               ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64)]),
    "tk_last_stats": (_INT, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                             ctypes.POINTER(_I64)]),
    "tk_cache_create": (_INT, [_P, _I64, ctypes.POINTER(_P)]),
    "tk_cache_free": (None, [_P]),
    "tk_cache_clear": (_INT, [_P, _P]),
    "tk_cache_stats": (_INT, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "tk_workspace_set_cache": (_INT, [_P, _P]),
    "tk_last_cache_stats": (_INT, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "tk_status_string": (ctypes.c_char_p, [_INT]),
    "tk_last_error": (ctypes.c_char_p, []),
}

_lib = None


class TkError(RuntimeError):
    def __init__(self, code, where):
        msg = _lib.tk_last_error().decode(errors="replace") if _lib is not None else ""
        name = _lib.tk_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {name} ({code}): {msg}")
        self.code = code


def lib_path():
    return _build.LIB


def load(build_if_missing=True):
    """Loads libtk.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libtk.so not built at {path}; run byte_level_bpe_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(code, where):
    if code != TK_OK:
        raise TkError(code, where)


def tk_load(rank_bytes, rank_off, rank_ids, n, spec_bytes, spec_off, spec_ids, n_spec,
            pattern_id=TK_PATTERN_CL100K):
    """Host pointers (ints) -> tokenizer handle (c_void_p)."""
    h = _P()
    check(load().tk_load(rank_bytes, rank_off, rank_ids, n, spec_bytes, spec_off, spec_ids,
                         n_spec, pattern_id, ctypes.byref(h)), "tk_load")
    return h


def tk_free(tok):
    if tok:
        load().tk_free(tok)


def tk_workspace_create(tok, max_bytes, max_segments):
    h = _P()
    check(load().tk_workspace_create(tok, max_bytes, max_segments, ctypes.byref(h)),
          "tk_workspace_create")
    return h


def tk_workspace_free(ws):
    if ws:
        load().tk_workspace_free(ws)


def tk_encode_segments(tok, ws, d_text, n_bytes, d_seg_off, d_allow_special, S, tiktoken_safe,
                       d_out_ids, out_capacity, d_out_offsets, stream, raise_on_error=True):
    """Device pointers (ints). Returns (status, n_ids)."""
    n = _I64(0)
    rc = load().tk_encode_segments(tok, ws, d_text, n_bytes, d_seg_off, d_allow_special, S,
                                   1 if tiktoken_safe else 0, d_out_ids, out_capacity,
                                   d_out_offsets, ctypes.byref(n), stream)
    if raise_on_error:
        check(rc, "tk_encode_segments")
    return rc, n.value


def tk_encode_segments_host(tok, ws, h_text, n_bytes, h_seg_off, h_allow_special, S,
                            tiktoken_safe, h_out_ids, out_capacity, h_out_offsets, stream,
                            raise_on_error=True):
    """Host pointers (ints). Returns (status, n_ids)."""
    n = _I64(0)
    rc = load().tk_encode_segments_host(tok, ws, h_text, n_bytes, h_seg_off, h_allow_special, S,
                                        1 if tiktoken_safe else 0, h_out_ids, out_capacity,
                                        h_out_offsets, ctypes.byref(n), stream)
    if raise_on_error:
        check(rc, "tk_encode_segments_host")
    return rc, n.value


def tk_decode(tok, ws, d_ids, n, d_out, cap, stream, raise_on_error=True):
    """Device pointers (ints). Returns (status, n_bytes)."""
    m = _I64(0)
    rc = load().tk_decode(tok, ws, d_ids, n, d_out, cap, ctypes.byref(m), stream)
    if raise_on_error:
        check(rc, "tk_decode")
    return rc, m.value


def tk_profile_enable(ws, on):
    check(load().tk_profile_enable(ws, 1 if on else 0), "tk_profile_enable")


def tk_profile_read(ws, max_kernels=24):
    """-> {kernel name: (total ms, launches)}"""
    names = (ctypes.c_char_p * max_kernels)()
    ms = (ctypes.c_double * max_kernels)()
    cnt = (_I64 * max_kernels)()
    k = load().tk_profile_read(ws, max_kernels, names, ms, cnt)
    if k < 0:
        check(k, "tk_profile_read")
    return {names[i].decode(): (ms[i], cnt[i]) for i in range(min(k, max_kernels))}


def tk_last_stats(ws):
    """-> (pre-tokens, ids, long pre-tokens) of the workspace's last encode."""
    a, b, c = _I64(0), _I64(0), _I64(0)
    check(load().tk_last_stats(ws, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
          "tk_last_stats")
    return a.value, b.value, c.value


def tk_decode_noalloc(tok, d_ids, n, d_out, cap, stream, raise_on_error=True):
    """Device pointers (ints); no workspace, no allocation. Returns (status, n_bytes)."""
    m = _I64(0)
    rc = load().tk_decode_noalloc(tok, d_ids, n, d_out, cap, ctypes.byref(m), stream)
    if raise_on_error:
        check(rc, "tk_decode_noalloc")
    return rc, m.value


class DecodeState(ctypes.Structure):
    """tk_decode_state: the bytes a streaming decode holds back between calls."""
    _fields_ = [("pending", ctypes.c_uint8 * 4), ("n_pending", ctypes.c_int32)]


def tk_decode_stream(tok, ws, state, d_ids, n, final, d_out, cap, stream, raise_on_error=True):
    """state: a DecodeState; device pointers (ints). Returns (status, n_bytes)."""
    m = _I64(0)
    rc = load().tk_decode_stream(tok, ws, ctypes.byref(state), d_ids, n, 1 if final else 0, d_out, cap,
                                 ctypes.byref(m), stream)
    if raise_on_error:
        check(rc, "tk_decode_stream")
    return rc, m.value


def tk_decode_segments(tok, ws, d_ids, n, d_id_off, S, d_out, cap, d_byte_off, stream, raise_on_error=True):
    """Device pointers (ints). Returns (status, total bytes)."""
    m = _I64(0)
    rc = load().tk_decode_segments(tok, ws, d_ids, n, d_id_off, S, d_out, cap, d_byte_off, ctypes.byref(m),
                                   stream)
    if raise_on_error:
        check(rc, "tk_decode_segments")
    return rc, m.value


def tk_cache_create(tok, max_bytes):
    h = _P()
    check(load().tk_cache_create(tok, max_bytes, ctypes.byref(h)), "tk_cache_create")
    return h


def tk_cache_free(cache):
    if cache:
        load().tk_cache_free(cache)


def tk_cache_clear(cache, stream):
    check(load().tk_cache_clear(cache, stream), "tk_cache_clear")


def tk_cache_stats(cache):
    """-> (entries, bytes, ids) held by the cache."""
    a, b, c = _I64(0), _I64(0), _I64(0)
    check(load().tk_cache_stats(cache, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "tk_cache_stats")
    return a.value, b.value, c.value


def tk_workspace_set_cache(ws, cache):
    check(load().tk_workspace_set_cache(ws, cache), "tk_workspace_set_cache")


def tk_last_cache_stats(ws):
    """-> (pieces found in the cache, pieces added) by the workspace's last encode."""
    a, b = _I64(0), _I64(0)
    check(load().tk_last_cache_stats(ws, ctypes.byref(a), ctypes.byref(b)), "tk_last_cache_stats")
    return a.value, b.value
