"""byte_level_bpe_gb300: byte-level BPE encoding on one GB300.

Python face of libtk (include/tk.h). The tokenizer is a tiktoken-style
encoding ("tiktoken Deep Dive", "An encoding is three objects, not a model"):
mergeable ranks (bytes -> rank = id), the cl100k split pattern and specials.
`encode_segments` takes ordered (text, allow_special) segments and returns
device tensors, in one native call ("Making Kimi K3 Tokenization 18x Faster
For Million Token Agentic Workloads", "One native call for the whole serving
path"; no Python lists of ids are ever built).

torch provides device memory and the current stream; every encode step runs
in libtk's CUDA kernels. Without a built libtk.so or a CUDA device the calls
raise.
"""
import numpy as np

from . import native
from .native import TkError  # noqa: F401

__all__ = ["Tokenizer", "TkError", "native"]


def _to_bytes(text):
    if isinstance(text, (bytes, bytearray, memoryview)):
        return bytes(text)
    # lone surrogates become U+FFFD ("tiktoken Deep Dive", "The byte floor":
    # a replaced lone surrogate round-trips as the replacement character)
    return text.encode("utf-8", errors="replace")


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("byte_level_bpe_gb300 needs a CUDA device (no CPU fallback)")
    return torch


class Tokenizer:
    """ranks: list of token byte strings (index = rank = id) or (bytes, id) pairs;
    specials: dict of str|bytes -> id."""

    def __init__(self, ranks, specials=None, pattern_id=native.TK_PATTERN_CL100K,
                 max_bytes=1 << 20, max_segments=4096):
        torch = _torch()
        if ranks and isinstance(ranks[0], tuple):
            toks = [t for t, _ in ranks]
            ids = [int(i) for _, i in ranks]
        else:
            toks = list(ranks)
            ids = list(range(len(toks)))
        rb = np.frombuffer(b"".join(toks), np.uint8)
        ro = np.zeros(len(toks) + 1, np.int64)
        np.cumsum([len(t) for t in toks], out=ro[1:])
        ri = np.asarray(ids, np.uint32)
        specials = specials or {}
        sbl = [_to_bytes(s) for s in specials]
        sb = np.frombuffer(b"".join(sbl) or b"\0", np.uint8)
        so = np.zeros(len(sbl) + 1, np.int64)
        if sbl:
            np.cumsum([len(s) for s in sbl], out=so[1:])
        si = np.asarray(list(specials.values()) or [0], np.int32)
        self.device = torch.device("cuda", torch.cuda.current_device())
        self._h = native.tk_load(rb.ctypes.data, ro.ctypes.data, ri.ctypes.data, len(toks),
                                 sb.ctypes.data, so.ctypes.data, si.ctypes.data, len(sbl),
                                 pattern_id)
        self.n_ranks = len(toks)
        self.specials = {(_to_bytes(k)): v for k, v in specials.items()}
        self._ws = None
        self._ws_cap = (0, 0)
        self.ensure_workspace(max_bytes, max_segments)

    def close(self):
        if getattr(self, "_ws", None):
            native.tk_workspace_free(self._ws)
            self._ws = None
        if getattr(self, "_cache", None):
            native.tk_cache_free(self._cache)
            self._cache = None
        if getattr(self, "_h", None):
            native.tk_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    @property
    def workspace(self):
        return self._ws

    def attach_cache(self, max_bytes=256 << 20):
        """A cross-call word cache for this tokenizer's encodes (None: detach)."""
        if getattr(self, "_cache", None):
            native.tk_workspace_set_cache(self._ws, None)
            native.tk_cache_free(self._cache)
            self._cache = None
        if max_bytes:
            self._cache = native.tk_cache_create(self._h, max_bytes)
            native.tk_workspace_set_cache(self._ws, self._cache)
        return self._cache

    def ensure_workspace(self, max_bytes, max_segments):
        """Grows the workspace (never inside an encode: allocation happens here)."""
        mb, ms = self._ws_cap
        if self._ws is not None and max_bytes <= mb and max_segments <= ms:
            return
        mb, ms = max(mb, max_bytes, 1), max(ms, max_segments, 1)
        if self._ws is not None:
            native.tk_workspace_free(self._ws)
            self._ws = None
        self._ws = native.tk_workspace_create(self._h, mb, ms)
        self._ws_cap = (mb, ms)
        if getattr(self, "_cache", None):
            native.tk_workspace_set_cache(self._ws, self._cache)

    # ------------------------------------------------------------------
    def pack(self, segments):
        """[(text, allow_special)] -> host (text uint8, seg_off int64, allow uint8)."""
        parts = [_to_bytes(t) for t, _ in segments]
        text = np.frombuffer(b"".join(parts), np.uint8) if parts else np.zeros(0, np.uint8)
        off = np.zeros(len(parts) + 1, np.int64)
        if parts:
            np.cumsum([len(p) for p in parts], out=off[1:])
        allow = np.asarray([1 if a else 0 for _, a in segments], np.uint8)
        return text, off, allow

    def encode_device(self, d_text, d_seg_off, d_allow, tiktoken_safe=True, out=None,
                      out_offsets=None, stream=None):
        """Device tensors in, device tensors out: (ids int32[n_ids], offsets int64[S+1])."""
        torch = _torch()
        n = int(d_text.numel())
        S = int(d_seg_off.numel()) - 1
        self.ensure_workspace(n, S)
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int32, device=self.device)
        if out_offsets is None:
            out_offsets = torch.empty(S + 1, dtype=torch.int64, device=self.device)
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        _, n_ids = native.tk_encode_segments(
            self._h, self._ws, d_text.data_ptr() if n else None, n, d_seg_off.data_ptr(),
            d_allow.data_ptr() if S else None, S, tiktoken_safe, out.data_ptr(), out.numel(),
            out_offsets.data_ptr(), st.cuda_stream)
        return out[:n_ids], out_offsets

    def encode_segments(self, segments, tiktoken_safe=True):
        """[(str|bytes, allow_special)] -> (ids int32 cuda tensor, offsets int64 cuda tensor)."""
        torch = _torch()
        text, off, allow = self.pack(segments)
        d_text = torch.from_numpy(text.copy()).to(self.device)
        d_off = torch.from_numpy(off).to(self.device)
        d_allow = torch.from_numpy(allow.copy() if allow.size else np.zeros(1, np.uint8)).to(self.device)
        return self.encode_device(d_text, d_off, d_allow, tiktoken_safe)

    def encode(self, text, allow_special=False, tiktoken_safe=True):
        ids, _ = self.encode_segments([(text, allow_special)], tiktoken_safe)
        return ids

    def encode_host(self, text, seg_off, allow, tiktoken_safe=True, out=None, out_offsets=None,
                    stream=None):
        """Host numpy arrays in and out through tk_encode_segments_host."""
        torch = _torch()
        n = int(text.size)
        S = int(seg_off.size) - 1
        self.ensure_workspace(n, S)
        if out is None:
            out = np.empty(max(n, 1), np.int32)
        if out_offsets is None:
            out_offsets = np.empty(S + 1, np.int64)
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        _, n_ids = native.tk_encode_segments_host(
            self._h, self._ws, text.ctypes.data, n, seg_off.ctypes.data, allow.ctypes.data, S,
            tiktoken_safe, out.ctypes.data, out.size, out_offsets.ctypes.data, st.cuda_stream)
        return out[:n_ids], out_offsets

    def decode_device(self, d_ids, out=None, stream=None):
        """Device int32 ids -> device uint8 bytes."""
        torch = _torch()
        n = int(d_ids.numel())
        self.ensure_workspace(n, 1)
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        if out is None:
            _, m = native.tk_decode(self._h, self._ws, d_ids.data_ptr() if n else None, n, None, 0,
                                    st.cuda_stream, raise_on_error=False)
            out = torch.empty(max(m, 1), dtype=torch.uint8, device=self.device)
        _, m = native.tk_decode(self._h, self._ws, d_ids.data_ptr() if n else None, n,
                                out.data_ptr(), out.numel(), st.cuda_stream)
        return out[:m]

    def decode_segments(self, d_ids, d_id_off, stream=None):
        """Device ids + id offsets[S+1] -> (device bytes, device byte offsets[S+1])."""
        torch = _torch()
        n = int(d_ids.numel())
        S = int(d_id_off.numel()) - 1
        self.ensure_workspace(max(n, 1), 1)
        st = stream if stream is not None else torch.cuda.current_stream(self.device)
        byte_off = torch.empty(S + 1, dtype=torch.int64, device=self.device)
        _, m = native.tk_decode_segments(self._h, self._ws, d_ids.data_ptr() if n else None, n,
                                         d_id_off.data_ptr(), S, None, 0, byte_off.data_ptr(),
                                         st.cuda_stream, raise_on_error=False)
        out = torch.empty(max(m, 1), dtype=torch.uint8, device=self.device)
        native.tk_decode_segments(self._h, self._ws, d_ids.data_ptr() if n else None, n, d_id_off.data_ptr(),
                                  S, out.data_ptr(), out.numel(), byte_off.data_ptr(), st.cuda_stream)
        return out[:m], byte_off

    def stream_decoder(self, stream=None):
        """Incremental decode: feed(ids) -> bytes that end on a character
        boundary (a trailing partial character waits for the next feed);
        finish() -> the bytes still held back."""
        return _StreamDecoder(self, stream)

    def decode(self, ids):
        torch = _torch()
        if not torch.is_tensor(ids):
            ids = torch.as_tensor(np.asarray(ids, np.int32))
        d = ids.to(self.device, dtype=torch.int32).contiguous()
        return self.decode_device(d).cpu().numpy().tobytes()


class _StreamDecoder:
    def __init__(self, tok, stream):
        self._tok = tok
        self._stream = stream
        self._state = native.DecodeState()

    def _call(self, ids, final):
        torch = _torch()
        tok = self._tok
        if not torch.is_tensor(ids):
            ids = torch.as_tensor(np.asarray(ids, np.int32))
        d = ids.to(tok.device, dtype=torch.int32).contiguous()
        n = int(d.numel())
        tok.ensure_workspace(max(n, 1), 1)
        st = self._stream if self._stream is not None else torch.cuda.current_stream(tok.device)
        rc, need = native.tk_decode_stream(tok._h, tok._ws, self._state, d.data_ptr() if n else None, n, final,
                                           None, 0, st.cuda_stream, raise_on_error=False)
        if rc not in (native.TK_OK, native.TK_E_CAPACITY):
            native.check(rc, "tk_decode_stream")
        out = torch.empty(max(need + 4, 1), dtype=torch.uint8, device=tok.device)
        _, m = native.tk_decode_stream(tok._h, tok._ws, self._state, d.data_ptr() if n else None, n, final,
                                       out.data_ptr(), out.numel(), st.cuda_stream)
        return out[:m].cpu().numpy().tobytes()

    def feed(self, ids):
        return self._call(ids, False)

    def finish(self):
        return self._call([], True)
