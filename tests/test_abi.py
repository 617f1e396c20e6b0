"""The C-ABI library builds, loads, and exports every function include/tk.h
declares (no GPU needed: only host-side calls)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "tk.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tk_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from byte_level_bpe_gb300 import native
    lib = native.load()
    declared = _declared()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
        assert name in native.SIGNATURES, name


def test_status_strings():
    from byte_level_bpe_gb300 import native
    lib = native.load()
    assert lib.tk_status_string(0) == b"ok"
    assert lib.tk_status_string(native.TK_E_UTF8) == b"invalid UTF-8"
    assert lib.tk_status_string(12345) == b"unknown status"


def _load(ranks, specials=None, pattern=1):
    from byte_level_bpe_gb300 import native
    lib = native.load()
    rb = np.frombuffer(b"".join(ranks) or b"\0", np.uint8)
    ro = np.zeros(len(ranks) + 1, np.int64)
    np.cumsum([len(t) for t in ranks], out=ro[1:])
    ri = np.arange(len(ranks), dtype=np.uint32)
    specials = specials or {}
    sb = np.frombuffer(b"".join(specials) or b"\0", np.uint8)
    so = np.zeros(len(specials) + 1, np.int64)
    if specials:
        np.cumsum([len(s) for s in specials], out=so[1:])
    si = np.asarray(list(specials.values()) or [0], np.int32)
    h = ctypes.c_void_p()
    rc = lib.tk_load(rb.ctypes.data, ro.ctypes.data, ri.ctypes.data, len(ranks), sb.ctypes.data,
                     so.ctypes.data, si.ctypes.data, len(specials), pattern, ctypes.byref(h))
    return rc, lib.tk_last_error().decode()


def test_table_validation_is_host_side():
    """tk_load rejects bad tables before touching the device."""
    from byte_level_bpe_gb300 import native
    floor = [bytes([b]) for b in range(256)]
    rc, msg = _load(floor[:255])
    assert rc == native.TK_E_TABLE and "byte floor" in msg
    rc, _ = _load(floor + [b"ab", b"ab"])
    assert rc == native.TK_E_TABLE
    rc, _ = _load(floor, {b"<|x|>": 65})
    assert rc == native.TK_E_TABLE
    rc, msg = _load(floor, {b"abab": 300})  # can overlap itself
    assert rc == native.TK_E_TABLE and "overlap" in msg
    rc, _ = _load(floor, {b"\xff": 300})  # not UTF-8
    assert rc == native.TK_E_TABLE
    rc, _ = _load(floor, pattern=3)  # patterns are 1 (cl100k) and 2 (cl100k with r50k digits)
    assert rc == native.TK_E_ARG


def test_no_cpu_fallback_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import byte_level_bpe_gb300 as tk
    with pytest.raises(RuntimeError):
        tk.Tokenizer([bytes([b]) for b in range(256)])


def test_product_never_imports_oracle():
    pkg = os.path.join(ROOT, "byte_level_bpe_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "bpe_oracle" not in src, f
