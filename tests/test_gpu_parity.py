"""GPU parity: the CUDA path's ids equal the CPU oracle's, element by element.

Every test calls the C ABI through the thin binding (byte_level_bpe_gb300)
and compares with the oracle on the same seeded inputs. Integer work:
bit-exact equality, no tolerance.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _gpu_ids(tk, segments, safe):
    ids, off = tk.encode_segments(segments, tiktoken_safe=safe)
    return ids.cpu().numpy(), off.cpu().numpy()


def _first_bad_segment(segments, g_ids, g_off, o_ids, o_off):
    for k, (s, allow) in enumerate(segments):
        a = g_ids[g_off[k]:g_off[k + 1]]
        b = o_ids[o_off[k]:o_off[k + 1]]
        if len(a) != len(b) or not np.array_equal(a, b):
            return f"segment {k} {s!r} allow={allow}: gpu {a.tolist()} oracle {b.tolist()}"
    return "no differing segment"


def _compare(tk, enc, segments, safe):
    g_ids, g_off = _gpu_ids(tk, segments, safe)
    o_ids, o_off = enc.encode_segments(segments, tiktoken_safe=safe)
    if len(g_ids) != len(o_ids) or not np.array_equal(g_off, o_off):
        raise AssertionError(f"{len(g_ids)} vs {len(o_ids)} ids; " +
                             _first_bad_segment(segments, g_ids, g_off, o_ids, o_off)[:3000])
    if not np.array_equal(g_ids, o_ids):
        k = int(np.argmax(g_ids != o_ids))
        raise AssertionError(f"first mismatch at id {k}: gpu {g_ids[k-3:k+4]} oracle {o_ids[k-3:k+4]}")
    assert np.array_equal(g_off, o_off)
    return g_ids


@pytest.fixture(scope="module")
def full_gpu(full_table):
    import byte_level_bpe_gb300 as tk
    return tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=1 << 24, max_segments=8192)


@pytest.fixture(scope="module")
def tiny_gpu(tiny_table):
    import byte_level_bpe_gb300 as tk
    return tk.Tokenizer(tiny_table, max_bytes=1 << 20)


def test_tiny_workload(tiny_gpu, tiny_enc):
    _compare(tiny_gpu, tiny_enc, [(workloads.tiny_input(), False)], False)


def test_full_table_workload(full_gpu, full_enc, full_table):
    text = workloads.prose_text(full_table, 1 << 20, seed=2)
    _compare(full_gpu, full_enc, [(text, False)], False)


def test_agentic_small(full_gpu, full_enc, full_table):
    segs = workloads.agentic_segments(full_table, seed=3, scale=0.05)
    _compare(full_gpu, full_enc, segs, True)


def test_agentic_full(full_gpu, full_enc, full_table):
    segs = workloads.agentic_segments(full_table, seed=3)
    assert max(len(s) for s, _ in segs) > 1_000_000
    _compare(full_gpu, full_enc, segs, True)


def test_multilingual(full_table):
    import byte_level_bpe_gb300 as tk
    ext = workloads.multilingual_table(full_table)
    ranks = [(t, i) for i, t in enumerate(full_table)] + ext
    enc = oracle.Encoding(ranks, workloads.SPECIALS)
    gpu = tk.Tokenizer(ranks, workloads.SPECIALS, max_bytes=1 << 24)
    text = workloads.multilingual_text(full_table)
    _compare(gpu, enc, [(text, False)], False)


def test_serving_scaled(full_gpu, full_enc, full_table):
    text, off = workloads.serving_batch(full_table, seed=5, total=8 << 20, n_req=128)
    segs = [(text[off[i]:off[i + 1]].tobytes(), False) for i in range(len(off) - 1)]
    _compare(full_gpu, full_enc, segs, False)


def test_serving_full_size(full_table, tmp_path):
    """The 256 MiB batch (4,096 requests) in the bench's launch configuration,
    every id compared with the oracle: requests are independent, so the
    oracle runs over groups of requests in a pool of host processes (spawned,
    not forked, since this process already holds a CUDA context)."""
    import multiprocessing as mp
    import os
    import byte_level_bpe_gb300 as tk
    text, off = workloads.serving_batch(full_table, seed=5)
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=len(text), max_segments=len(off))
    d_text = torch.from_numpy(text).cuda()
    d_off = torch.from_numpy(off).cuda()
    d_allow = torch.zeros(len(off) - 1, dtype=torch.uint8, device="cuda")
    ids, g_off = gpu.encode_device(d_text, d_off, d_allow, tiktoken_safe=False)
    ids = ids.cpu().numpy()
    g_off = g_off.cpu().numpy()
    assert g_off[-1] == len(ids) and len(ids) > 100_000_000
    # properties at full size: ids decode back to the text
    assert gpu.decode(torch.from_numpy(ids)) == text.tobytes()
    gpu.close()
    del d_text
    path = str(tmp_path / "c5")
    np.save(path + "_text.npy", text)
    np.save(path + "_off.npy", off)
    np.save(path + "_ids.npy", ids)
    np.save(path + "_goff.npy", g_off)
    S = len(off) - 1
    # groups of consecutive requests of about 4 MiB
    groups, lo = [], 0
    while lo < S:
        hi = lo + 1
        while hi < S and off[hi + 1] - off[lo] <= 4 << 20:
            hi += 1
        groups.append((path, lo, hi))
        lo = hi
    import oracle_pool
    ctx = mp.get_context("spawn")
    with ctx.Pool(max(1, min(32, os.cpu_count() or 1)), initializer=oracle_pool.init,
                  initargs=(full_table,)) as pool:
        errors = [e for e in pool.imap_unordered(oracle_pool.check_requests, groups) if e]
    assert not errors, errors[:5]


# ---------------------------------------------------------------------------
# Edge cases

ALPHABET = ["a", "s", "L", "1", " ", "\n", "\r", "\t", "'", ".", "é", "ा", "\U0001F600",
            " ", "\x00", "ſ", "१", "v", "e", "r", "l", "T", "<|endoftext|>", "中"]


def test_special_cut_by_chunking_is_text(full_gpu, full_enc):
    """tiktoken_safe cuts before specials are matched: a special that a 25k-run
    cut or a 400k window cut falls inside stays ordinary text, while the same
    special clear of any cut is its id ("One native call for the whole serving
    path": the legacy path chunked the text, then encoded each chunk)."""
    eot = "<|endoftext|>"
    eot_id = workloads.SPECIALS[eot]
    run_cut = "x" * 24_995 + eot + " tail"            # the run's 25,000th character is inside it
    prose = ("ab cd " * 70_000)[:399_995]              # runs stay short; character 400,000 is inside it
    window_cut = prose + eot + " tail"
    clear = "x" * 100 + eot + " tail"
    for text in (run_cut, window_cut):
        g = _compare(full_gpu, full_enc, [(text, True)], True)
        assert eot_id not in set(g.tolist())
        _compare(full_gpu, full_enc, [(text, True)], False)  # unchunked: the special is matched
    g = _compare(full_gpu, full_enc, [(clear, True), (run_cut, True), (clear, True)], True)
    assert (g == eot_id).sum() == 2


def test_random_segments_fuzz(full_gpu, full_enc):
    rng = np.random.default_rng(11)
    segs = []
    for i in range(3000):
        L = int(rng.integers(0, 40))
        s = "".join(ALPHABET[j] for j in rng.integers(0, len(ALPHABET), size=L))
        segs.append((s, bool(rng.integers(0, 2))))
    _compare(full_gpu, full_enc, segs, False)
    _compare(full_gpu, full_enc, segs, True)


@pytest.mark.parametrize("n", [0, 1, 2, 15, 16, 17, 4095, 4096, 4097, 8191, 8193, 12288 + 5])
def test_ragged_sizes(full_gpu, full_enc, full_table, n):
    text = workloads.prose_text(full_table, n + 10, seed=n)[:n]
    while n and (text[-1] & 0xC0) == 0x80:
        text = text[:-1]
    _compare(full_gpu, full_enc, [(text, False)], False)


def test_empty_segments(full_gpu, full_enc):
    segs = [("", True), ("", False), ("ab cd", False), ("", True), ("<|endoftext|>", True), ("", False)]
    _compare(full_gpu, full_enc, segs, True)
    _compare(full_gpu, full_enc, [("", False)], False)


def test_tile_boundary_runs(full_gpu, full_enc):
    """Runs that straddle 4 KiB tiles: digits (mod-3 grouping carried across
    tiles), white space with CR/LF, other runs followed by CR/LF, specials,
    contractions and multi-byte characters at the boundary."""
    cases = []
    for off in range(4080, 4100):
        pad = "x" * (off - 3)
        cases.append(pad + " " + "1234567890" * 3 + " end")
        cases.append(pad + "..\n\n   word")
        cases.append(pad + "\n\n    \n   \tcode")
        cases.append(pad + "it's 'll 'VE don't")
        cases.append(pad + "é中\U0001F600ſ'ſ")
        cases.append(pad + "<|endoftext|><|fim_prefix|>")
        cases.append(pad + "   \n")
    for c in cases:
        _compare(full_gpu, full_enc, [(c, True)], False)
        _compare(full_gpu, full_enc, [(c, False)], True)


def test_long_digit_and_space_runs(full_gpu, full_enc):
    for text in ["7" * 20011, " " * 30000 + "x", "\n" * 9000 + "  " + "a" * 9000,
                 "." * 5000 + "\n" * 5000 + " " * 5000 + "z", " " * 70001, "ab" * 40000]:
        _compare(full_gpu, full_enc, [(text, False)], False)
        _compare(full_gpu, full_enc, [(text, True)], True)


def test_safe_chunking_window(full_gpu, full_enc):
    text = "é" * 399_999 + "中" + "\U0001F600" * 5 + "x" * 10 + " " * 60_000 + "<|endoftext|>" + "y" * 26_000
    _compare(full_gpu, full_enc, [(text, True)], True)
    _compare(full_gpu, full_enc, [(text, False)], True)


def test_invalid_utf8(full_gpu):
    import byte_level_bpe_gb300 as tk
    for bad, pos in [(b"ab\xffcd", 2), (b"abc\xc0\x80", 3), (b"\xed\xa0\x80", 0), (b"xy\xe4\xb8", 2),
                     (b"\x80", 0), (b"a" * 5000 + b"\xf5", 5000)]:
        with pytest.raises(tk.TkError) as ei:
            full_gpu.encode(bad)
        assert ei.value.code == tk.native.TK_E_UTF8
        assert f"byte {pos}" in str(ei.value)


def test_capacity_error_reports_count(full_gpu, full_enc):
    import byte_level_bpe_gb300 as tk
    text = b"hello world, this is a test"
    exp = full_enc.encode(text)
    d_text = torch.frombuffer(bytearray(text), dtype=torch.uint8).cuda()
    d_off = torch.tensor([0, len(text)], dtype=torch.int64, device="cuda")
    d_allow = torch.zeros(1, dtype=torch.uint8, device="cuda")
    out = torch.empty(2, dtype=torch.int32, device="cuda")
    with pytest.raises(tk.TkError) as ei:
        full_gpu.encode_device(d_text, d_off, d_allow, False, out=out)
    assert ei.value.code == tk.native.TK_E_CAPACITY
    rc, n = tk.native.tk_encode_segments(full_gpu.handle, full_gpu.workspace, d_text.data_ptr(),
                                         len(text), d_off.data_ptr(), d_allow.data_ptr(), 1, 0,
                                         out.data_ptr(), 2, d_off.data_ptr() if False else
                                         torch.empty(2, dtype=torch.int64, device="cuda").data_ptr(),
                                         torch.cuda.current_stream().cuda_stream, raise_on_error=False)
    assert rc == tk.native.TK_E_CAPACITY and n == len(exp)


def test_unaligned_text_pointer(full_gpu, full_enc, full_table):
    text = workloads.prose_text(full_table, 20000, seed=4)
    buf = torch.frombuffer(bytearray(b"z" + text), dtype=torch.uint8).cuda()
    d_text = buf[1:]
    assert d_text.data_ptr() % 16 != 0
    d_off = torch.tensor([0, len(text)], dtype=torch.int64, device="cuda")
    d_allow = torch.zeros(1, dtype=torch.uint8, device="cuda")
    ids, _ = full_gpu.encode_device(d_text, d_off, d_allow, False)
    assert np.array_equal(ids.cpu().numpy(), full_enc.encode(text))


def test_decode_round_trip_and_bad_id(full_gpu):
    import byte_level_bpe_gb300 as tk
    s = "NUL:\x00 emoji:\U0001F600 CJK:中文 replaced:\ud800 end <|endoftext|>"
    ids, _ = full_gpu.encode_segments([(s, True)])
    assert full_gpu.decode(ids) == s.encode("utf-8", "replace")
    with pytest.raises(tk.TkError) as ei:
        full_gpu.decode(np.array([65, 100256], np.int32))  # 100256 is in the reserved gap
    assert ei.value.code == tk.native.TK_E_BADID


def test_host_buffer_entry_point(full_gpu, full_enc, full_table):
    segs = workloads.agentic_segments(full_table, seed=7, scale=0.01)
    text, off, allow = workloads.pack_segments(segs)
    ids, offs = full_gpu.encode_host(np.ascontiguousarray(text), off, allow, tiktoken_safe=True)
    o_ids, o_off = full_enc.encode_segments(segs, tiktoken_safe=True)
    assert np.array_equal(ids, o_ids) and np.array_equal(offs, o_off)


def test_two_calls_in_a_row_reuse_workspace(full_gpu, full_enc, full_table):
    a = workloads.prose_text(full_table, 50000, seed=8)
    b = workloads.prose_text(full_table, 30000, seed=9)
    for t in (a, b, a):
        _compare(full_gpu, full_enc, [(t, False)], False)


def test_long_white_space_walks(full_gpu, full_enc):
    """CR/LF followed by white space whose run leaves the tile's window: the
    run may end in text, at a special (a piece start), at a chunk cut or at
    the text end."""
    tails = ["<|endoftext|>", "x", "", "  y", "\n\n z"]
    segs = []
    for pad in (3, 4000, 4090, 8150):
        for run in (70, 200, 1000, 5000):
            for tail in tails:
                body = "a" * pad + "\n" + " " * run + "\n " + " \t" * (run // 4) + tail
                segs.append((body, True))
                segs.append((body, False))
    _compare(full_gpu, full_enc, segs, False)
    _compare(full_gpu, full_enc, segs, True)
    long_run = "q\n" + " " * 60_000 + "<|endoftext|>" + "\n" + " " * 30_000 + "w"
    _compare(full_gpu, full_enc, [(long_run, True)], True)
    _compare(full_gpu, full_enc, [(long_run, True)], False)


def test_host_buffer_pipelined(full_table, full_enc):
    """A host call large enough to be cut into batches at segment boundaries:
    ids and offsets equal the one-shot device call's, sampled segments equal
    the oracle's, and errors keep their whole-call meaning."""
    import byte_level_bpe_gb300 as tk
    text, off = workloads.serving_batch(full_table, seed=11, total=40 << 20, n_req=600)
    segs = []
    for r in range(len(off) - 1):
        body = text[off[r]:off[r + 1]].tobytes()
        if r % 7 == 0:
            body = b"<|endoftext|>" + body
        segs.append((body, r % 2 == 0))
    h_text, h_off, h_allow = workloads.pack_segments(segs)
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=len(h_text), max_segments=len(segs))
    ids_h, off_h = gpu.encode_host(np.ascontiguousarray(h_text), h_off, h_allow, tiktoken_safe=True)
    ids_d, off_d = gpu.encode_device(torch.from_numpy(h_text).cuda(), torch.from_numpy(h_off).cuda(),
                                     torch.from_numpy(h_allow).cuda(), tiktoken_safe=True)
    assert np.array_equal(off_h, off_d.cpu().numpy())
    assert np.array_equal(ids_h, ids_d.cpu().numpy())
    rng = np.random.default_rng(1)
    for r in sorted(set(rng.choice(len(segs), size=12, replace=False).tolist()) | {0, len(segs) - 1}):
        o_ids, _ = full_enc.encode_segments([segs[r]], tiktoken_safe=True)
        assert np.array_equal(ids_h[off_h[r]:off_h[r + 1]], o_ids), r
    # an invalid byte late in the text: reported at its position in the whole call
    bad = h_text.copy()
    pos = int(h_off[len(segs) - 3]) + 5
    bad[pos] = 0xFF
    with pytest.raises(tk.TkError) as ei:
        gpu.encode_host(bad, h_off, h_allow, tiktoken_safe=True)
    assert ei.value.code == tk.native.TK_E_UTF8 and f"byte {pos}" in str(ei.value)
    # too small an output: the capacity error carries the full count
    out = np.empty(len(ids_h) - 1, np.int32)
    out_off = np.empty(len(segs) + 1, np.int64)
    rc, n = tk.native.tk_encode_segments_host(
        gpu.handle, gpu.workspace, h_text.ctypes.data, len(h_text), h_off.ctypes.data,
        h_allow.ctypes.data, len(segs), 1, out.ctypes.data, out.size, out_off.ctypes.data,
        torch.cuda.current_stream().cuda_stream, raise_on_error=False)
    assert rc == tk.native.TK_E_CAPACITY and n == len(ids_h)
    # and the workspace still encodes correctly afterwards
    ids2, off2 = gpu.encode_host(np.ascontiguousarray(h_text), h_off, h_allow, tiktoken_safe=True)
    assert np.array_equal(ids2, ids_h) and np.array_equal(off2, off_h)
    gpu.close()


def test_cluster_merged_pieces(full_gpu, full_enc):
    """Pre-tokens long enough for the CTA-cluster merge (over 16 KiB), with
    small alphabets so that many ranks and long merge chains occur; one piece
    appears twice (the copy takes the first one's ids)."""
    rng = np.random.default_rng(12)
    pieces = [("".join(rng.choice(list(a), n))).encode() for n, a in
              [(16385, "ab"), (20000, "abc"), (30000, "etaoin"), (80000, "esr"), (17000, "a")]]
    segs = [(p, False) for p in pieces] + [(b" " + pieces[2], False), (pieces[1], False)]
    _compare(full_gpu, full_enc, segs, False)
    _compare(full_gpu, full_enc, segs, True)


def test_mid_length_pieces(full_gpu, full_enc):
    """Pre-tokens of 17..1024 bytes (merged per warp outside the tile kernel),
    around the one- and two-slot register limits (32 and 64 bytes), repeated
    so that copies take their owner's ids, mixed with short words."""
    rng = np.random.default_rng(21)
    parts = []
    for n in [17, 18, 31, 32, 33, 47, 63, 64, 65, 100, 513, 1024]:
        for alpha in ["ab", "etaoinshr", "abcdefghijklmnopqrstuvwxyz"]:
            w = "".join(rng.choice(list(alpha), n))
            parts += [" " + w[1:], w, " " + w[1:]]
    for n in [17, 40, 64, 65, 96, 97, 128, 129, 300]:
        parts += ["-" * n, "=" * n, "a" * n, "x" + " " * n + "y"]
    rng.shuffle(parts)
    text = " ".join(parts).encode()
    segs = [(text[i:i + 5000], False) for i in range(0, len(text), 5000)]
    _compare(full_gpu, full_enc, segs, False)


def test_token_that_does_not_encode_to_itself():
    """A table may hold a token that the merge loop never builds from its own
    bytes: with bc < ab < cd < abcd, "abcd" merges bc first and stops at
    [a, bc, d].  Such a token must not be used as a whole-piece shortcut."""
    import byte_level_bpe_gb300 as tk
    table = [bytes([i]) for i in range(256)] + [b"bc", b"ab", b"cd", b"abcd", b"wxyz", b"wx", b"yz"]
    # wxyz (rank 260) is unreachable too: wx (261) and yz (262) come later
    enc = oracle.Encoding(table, {})
    gpu = tk.Tokenizer(table, {}, max_bytes=1 << 16, max_segments=4)
    text = "abcd abcd wxyz abcdabcd wxyzwxyz ab cd bc"
    g_ids, _ = gpu.encode_segments([(text, False)], tiktoken_safe=False)
    o_ids = enc.encode(text.encode())
    assert np.array_equal(g_ids.cpu().numpy(), o_ids)
    assert list(enc.encode(b"abcd")) == [ord("a"), 256, ord("d")]
    gpu.close()


def test_r50k_digit_clause(full_table):
    """The split pattern with r50k's digit clause: the agentic prompt (JSON
    numbers, hex ids), digit/space-heavy random segments, and digit runs that
    cross tiles and exceed the long-piece thresholds."""
    import byte_level_bpe_gb300 as tk
    enc = oracle.Encoding(full_table, workloads.SPECIALS, pattern=oracle.PATTERN_R50K_DIGITS)
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, pattern_id=tk.native.TK_PATTERN_R50K_DIGITS,
                       max_bytes=1 << 24, max_segments=8192)
    _compare(gpu, enc, workloads.agentic_segments(full_table, seed=3, scale=0.25), True)
    rng = np.random.default_rng(23)
    alpha = ["1", "9", "0", " ", "  ", "\t", "\n", "a", "x", "$", ".", "१", "٣", " 12", "'s", "\r\n"]
    segs = []
    for _ in range(1500):
        L = int(rng.integers(0, 40))
        segs.append(("".join(alpha[i] for i in rng.integers(0, len(alpha), size=L)), bool(rng.integers(0, 2))))
    _compare(gpu, enc, segs, False)
    _compare(gpu, enc, segs, True)
    digits = "".join(str(d) for d in rng.integers(0, 10, size=70000))
    long_segs = [(digits[:5000], False), (" " + digits[:40000], False), ("a " + digits, False),
                 (("x " + digits[:3000]) * 5, False), (" " * 3 + digits[:100], False)]
    _compare(gpu, enc, long_segs, False)
    _compare(gpu, enc, long_segs, True)
    gpu.close()


def test_tile_tables_dense_and_ragged(full_gpu, full_enc):
    """Pieces of 5..16 bytes (merged over the whole grid) and of 1..4 bytes
    (merged in the tile kernel) at every offset around tile ends and the text
    end; a tile packed with 5-byte pieces (the most table entries a tile can
    hold); segment starts inside such tiles, empty ones included; specials
    next to mid pieces; a piece of over 8192 ids in a tile whose other
    pieces are mid pieces (the per-part copy path)."""
    rng = np.random.default_rng(31)
    letters = list("etaoinshrdlucmfwypvbgkqjxz")
    segs = []
    # every length 1..18 ending at every offset around the first tile end
    for L in range(1, 19):
        for shift in range(-3, 4):
            pre = 4096 - L + shift
            filler = (" ab" * ((pre // 3) + 1))[:pre]
            w = "".join(rng.choice(letters, L - 1))
            segs.append((filler + " " + w + " x", False))
            segs.append((filler + " " + w, False))  # ends at the text end
    # dense: " abcd" is a 5-byte piece, 819 of them per tile
    dense = " abcd" * 2500
    segs.append((dense, False))
    cuts = sorted(int(c) for c in rng.integers(0, len(dense), size=40))
    prev = 0
    for c in cuts + [len(dense)]:
        segs.append((dense[prev:c], False))
        segs.append(("", False))
        prev = c
    # specials (13 and 15 bytes) between mid pieces
    sp = list(workloads.SPECIALS)
    segs.append(((" hello" + sp[0] + " worldly" + sp[-1] + " abcdefghij") * 50, True))
    # over 8192 ids in one piece, after mid pieces in the same tile
    big = "".join(rng.choice(letters, 30000))
    segs.append((" mixture parsing tokens" * 20 + " " + big + " tail", False))
    _compare(full_gpu, full_enc, segs, False)
    _compare(full_gpu, full_enc, segs, True)


def test_mid_word_cache_keys(full_gpu, full_enc):
    """The mid-piece word cache (used by calls of 8 MiB or more) keys pieces
    of 5..16 bytes by their bytes, zero-padded, and their length: pieces that
    differ only by trailing NUL bytes, or whose second key word is zero, must
    stay apart; hot words repeated hundreds of thousands of times share one
    merge.  9 MiB in 1,300 segments."""
    base = ["!!!!!", "!!!!!\0", "!!!!!\0\0", "!!!!!!!!", "!!!!!!!!\0", "!!!!!!!!\0\0",
            "!!!!!!!!\0!", "!!!!!!!!!!!!!!!\0", "\0\0\0\0\0", "\0\0\0\0\0\0\0\0\0",
            "--------", "--------\0", "#$%&#$%&#$%&", "#$%&#$%&#$%&\0"]
    rng = np.random.default_rng(41)
    words = [" information", " tokenizer", " encodings", "abcdefgh", " merges", " the", " of"]
    parts = [base[i] for i in rng.integers(0, len(base), size=120000)]
    parts += [words[i] for i in rng.integers(0, len(words), size=900000)]
    rng.shuffle(parts)
    text = "\n".join(parts)
    assert len(text) >= 8 << 20
    segs = [(text[i:i + 7300], False) for i in range(0, len(text), 7300)]
    _compare(full_gpu, full_enc, segs, False)


def test_big_mixed_white_space_pieces(full_gpu, full_enc):
    """Pre-tokens of 1,025-26,000 bytes of mixed white space (spaces, tabs and
    their boundaries, which no token of the table holds), runs ending in CR/LF
    and a long letter/white-space mix: the exact rounds of the big-piece merge
    against the oracle's parts loop."""
    rng = np.random.default_rng(23)
    segs = []
    for n in (1030, 1500, 4000, 9000, 17000, 26000):
        for mix in ((" ", "\t"), (" ", " ", " ", "\t", "\t\t"), (" ", "\t", " \t ")):
            parts = []
            while sum(len(p) for p in parts) < n:
                parts.append(mix[int(rng.integers(0, len(mix)))] * int(rng.integers(1, 40)))
            run = "".join(parts)[:n]
            segs.append(("x" + run + "y", False))
            segs.append((run + "\n", False))
    segs.append(("a" + " \t" * 5 + " " * 2000 + "b", False))
    segs.append(("q" + "ab" * 900 + " " + "\t" * 1200, False))
    _compare(full_gpu, full_enc, segs, False)
    _compare(full_gpu, full_enc, segs, True)


def test_big_pieces_chunk_edges(full_gpu, full_enc):
    """Pre-tokens of 1,025-32,768 bytes merged by one CTA over warp-owned
    chunks: lengths around the chunk and shared-memory sizes (one repeated
    letter), runs of pairs of one rank crossing chunk ends ("ab..."), and
    random letters of a small alphabet, whose rounds merge a few pairs each
    and stop early at lower-ranked neighbour pairs."""
    rng = np.random.default_rng(29)
    segs = []
    for n in (1025, 1056, 1057, 2049, 4097, 22990, 23010, 32768):
        segs.append((" " + "a" * (n - 1), False))
    for n in (1100, 3001, 7777):
        segs.append(("ab" * (n // 2) + "a", False))
        segs.append(("abc" * (n // 3), False))
    for alpha, n in (("etaoin", 1100), ("etaoin", 3000), ("ab", 4000), ("aeiost", 9000)):
        letters = np.array(list(alpha))
        segs.append(("".join(letters[rng.integers(0, len(letters), n)]), False))
    _compare(full_gpu, full_enc, segs, False)


def _shuffled_ab_table(seed):
    """The 256 bytes, then tokens over {a, b} of 2-8 bytes built from pairs of
    earlier tokens, in a shuffled rank order: many tokens then have an
    extension (a token a||x or x||b) ranked below them, so the exact rounds'
    stop rule fires."""
    rng = np.random.default_rng(seed)
    toks = [b"a", b"b"]
    seen = set(toks)
    while len(toks) < 300:
        t = toks[int(rng.integers(0, len(toks)))] + toks[int(rng.integers(0, len(toks)))]
        if len(t) <= 8 and t not in seen:
            seen.add(t)
            toks.append(t)
    multi = toks[2:]
    order = rng.permutation(len(multi))
    return [bytes([i]) for i in range(256)] + [multi[k] for k in order]


def test_long_pieces_stop_rule():
    """Pre-tokens of random a/b letters over a table with shuffled ranks, at
    the lengths of every merge path of the long pieces (a warp's list: 17-128
    bytes; a warp's rounds: 129-1,024; a CTA over chunks: 1,025-32,768; an 8-CTA
    cluster: longer): rounds stop at merges that create lower-ranked neighbour
    pairs."""
    import byte_level_bpe_gb300 as tk
    table = _shuffled_ab_table(31)
    rank = {t: i for i, t in enumerate(table)}
    low = sum(1 for t, r in rank.items() for k in range(1, len(t))
              if t[:k] in rank and t[k:] in rank and (r < rank[t[k:]] or r < rank[t[:k]]))
    assert low > 20  # the table exercises the stop rule
    enc = oracle.Encoding(table, {})
    gpu = tk.Tokenizer(table, {}, max_bytes=1 << 18, max_segments=64)
    rng = np.random.default_rng(37)
    segs = []
    for n in (17, 40, 77, 100, 128, 200, 700, 1100, 2500, 6000, 23500, 33000):
        segs.append(("".join(np.array(["a", "b"])[rng.integers(0, 2, n)]), False))
    segs.append(("ab" * 3000, False))
    segs.append(("a" * 5000 + "b" * 3000, False))
    _compare(gpu, enc, segs, False)
    gpu.close()


def _repeat_calls(gpu, enc, segments, safe, other):
    """The same call four times on the same buffers (direct, captured into a
    graph, replayed twice), an unrelated call, then the first again: every
    result equals the oracle's (the output is poisoned before each call)."""
    import torch
    text, off, allow = gpu.pack(segments)
    d_text = torch.from_numpy(text.copy()).cuda()
    d_off = torch.from_numpy(off).cuda()
    d_allow = torch.from_numpy(allow.copy()).cuda()
    out = torch.empty(max(text.size, 1), dtype=torch.int32, device="cuda")
    out_off = torch.empty(off.size, dtype=torch.int64, device="cuda")
    o_ids, o_off = enc.encode_segments(segments, tiktoken_safe=safe)
    for k in range(6):
        if k == 4:
            _compare(gpu, enc, other, safe)
            continue
        out.fill_(-1)
        out_off.fill_(-1)
        ids, offs = gpu.encode_device(d_text, d_off, d_allow, safe, out=out, out_offsets=out_off)
        assert np.array_equal(ids.cpu().numpy(), o_ids), f"call {k}"
        assert np.array_equal(offs.cpu().numpy(), o_off), f"call {k}"


def test_repeated_call_graph_small(full_gpu, full_enc, full_table):
    """A repeated call under 16 MiB (tiktoken_safe: chunk scans, the long
    pieces' streams) replayed from its captured graph."""
    segs = workloads.agentic_segments(full_table, seed=3, scale=0.05)
    other = [(workloads.prose_text(full_table, 20000, seed=12), False)]
    _repeat_calls(full_gpu, full_enc, segs, True, other)


def test_repeated_call_graph_large(full_table, full_enc):
    """A repeated call of 16 MiB (the mid pieces' stream and word cache too):
    calls this large launch directly each time, with the same results."""
    import byte_level_bpe_gb300 as tk
    text, off = workloads.serving_batch(full_table, seed=5, total=16 << 20, n_req=512)
    segs = [(bytes(text[off[i]:off[i + 1]]), False) for i in range(len(off) - 1)]
    gpu = tk.Tokenizer(full_table, workloads.SPECIALS, max_bytes=16 << 20, max_segments=1024)
    other = [(workloads.prose_text(full_table, 20000, seed=13), False)]
    _repeat_calls(gpu, full_enc, segs, False, other)
    gpu.close()
