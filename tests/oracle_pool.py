"""Worker functions for comparing a large GPU encode with the oracle in a
pool of spawned host processes (test infrastructure; no torch import, so the
workers start quickly and never touch CUDA)."""
import numpy as np

_ENC = None


def init(table):
    global _ENC
    import oracle
    import workloads
    _ENC = oracle.Encoding(table, workloads.SPECIALS)


def check_requests(args):
    """Encodes requests lo..hi-1 (allow_special = 0, no chunking) with the
    oracle and compares ids and offsets with the GPU's, both read from .npy
    files the parent wrote. Returns None, or a description of the mismatch."""
    path, lo, hi = args
    text = np.load(path + "_text.npy", mmap_mode="r")
    off = np.load(path + "_off.npy")
    ids = np.load(path + "_ids.npy", mmap_mode="r")
    g_off = np.load(path + "_goff.npy")
    sub_off = off[lo:hi + 1] - off[lo]
    exp, exp_off = _ENC.encode_arrays(np.ascontiguousarray(text[off[lo]:off[hi]]), sub_off,
                                      np.zeros(hi - lo, np.uint8), hi - lo, False)
    got_off = g_off[lo:hi + 1] - g_off[lo]
    if not np.array_equal(got_off, exp_off):
        k = int(np.argmax(got_off != exp_off))
        return f"offsets differ first at request {lo + k}"
    got = np.asarray(ids[g_off[lo]:g_off[hi]])
    if not np.array_equal(got, exp):
        k = int(np.argmax(got != exp)) if len(got) == len(exp) else -1
        return f"ids of requests {lo}..{hi - 1} differ (first at {k})"
    return None
