"""Seeded generators for the five synthetic workloads (numpy only).

Nothing here splits, merges or chunks text: the generators only choose random
token strings and lay out bytes. Every function takes a seed (numpy
default_rng) and is deterministic for it.
"""
from collections import defaultdict

import numpy as np

KiB = 1024
MiB = 1024 * 1024

# Specials with the ids of the cl100k-shaped table ("tiktoken Deep Dive",
# "Special tokens ...": <|endoftext|> 100257, three FIM markers, <|endofprompt|>
# 100276). The FIM names are not printed on the page; these are the reading.
SPECIALS = {
    "<|endoftext|>": 100257,
    "<|fim_prefix|>": 100258,
    "<|fim_middle|>": 100259,
    "<|fim_suffix|>": 100260,
    "<|endofprompt|>": 100276,
}

LOWER = b"abcdefghijklmnopqrstuvwxyz"
UPPER = b"ABCDEFGHIJKLMNOPQRSTUVWXYZ"
PUNCT = b"!\"#$%&'()*+,-./:;<=>?@[\\]^_`{|}~"
PROSE_PUNCT = [b".", b",", b";", b":", b"!", b"?", b'"', b"'", b"(", b")", b"-"]


def _zipf_cdf(n, s):
    w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def _zipf_draw(rng, cdf, size):
    return np.minimum(np.searchsorted(cdf, rng.random(size)), len(cdf) - 1)


def _digits(rng, n):
    return bytes(rng.integers(0x30, 0x3A, size=n).astype(np.uint8))


# --------------------------------------------------------------------------
# Tiny workload: 20,000 lowercase words, Zipf(1.1) slots.

def _tiny_words(seed=100):
    rng = np.random.default_rng(seed)
    words, seen = [], set()
    while len(words) < 20000:
        L = int(rng.integers(2, 11))
        w = bytes(rng.integers(0x61, 0x7B, size=L).astype(np.uint8))
        if w not in seen:
            seen.add(w)
            words.append(w)
    return words


def _slot_text(rng, words, cdf, n_bytes):
    """Words joined by single spaces; 5% punctuation attached to the previous
    word, 3% digit runs of 1-12 digits, 2% newlines."""
    out, size, after_nl = [], 0, True
    while size < n_bytes:
        kinds = rng.choice(4, size=4096, p=[0.90, 0.05, 0.03, 0.02])
        wi = _zipf_draw(rng, cdf, 4096)
        pk = rng.integers(0, len(PROSE_PUNCT), size=4096)
        dl = rng.integers(1, 13, size=4096)
        for k in range(4096):
            kind = kinds[k]
            if kind == 0:
                p = words[wi[k]] if after_nl else b" " + words[wi[k]]
            elif kind == 1:
                p = PROSE_PUNCT[pk[k]]
            elif kind == 2:
                p = (b"" if after_nl else b" ") + _digits(rng, int(dl[k]))
            else:
                p = b"\n"
            after_nl = kind == 3
            out.append(p)
            size += len(p)
            if size >= n_bytes:
                break
    return b"".join(out)[:n_bytes]


def tiny_corpus(n_bytes=2 * MiB, seed=101):
    """The 2 MiB training corpus of the tiny workload."""
    words = _tiny_words()
    return _slot_text(np.random.default_rng(seed), words, _zipf_cdf(len(words), 1.1), n_bytes)


def tiny_input(n_bytes=64 * KiB, seed=102):
    """The 64 KiB input of the tiny workload (same generator, another seed)."""
    words = _tiny_words()
    return _slot_text(np.random.default_rng(seed), words, _zipf_cdf(len(words), 1.1), n_bytes)


# --------------------------------------------------------------------------
# Full-size table: 100,256 ranks shaped like cl100k ("tiktoken Deep Dive",
# "The byte floor": 256 / 3,830 / 11,939 / 15,057 tokens of lengths 1-4,
# tapering to a 128-byte maximum).

def _length_counts():
    counts = {2: 3830, 3: 11939, 4: 15057}
    q = 69174 / (15057 + 69174)
    for L in range(5, 129):
        counts[L] = max(1, int(round(15057 * q ** (L - 4)))) if L <= 56 else 1
    counts[5] -= sum(counts.values()) - (100256 - 256)
    assert sum(counts.values()) == 100256 - 256
    return counts


def full_table(seed=2):
    """100,256 mergeable tokens; index = rank = id. Every token of length >= 2 is
    the concatenation of two lower-rank tokens (short, early pieces preferred)."""
    rng = np.random.default_rng(seed)
    toks = [bytes([b]) for b in range(256)]
    have = set(toks)
    pool = defaultdict(lambda: defaultdict(list))  # pool[cat][len] -> [bytes]
    for c in LOWER:
        pool["lower"][1].append(bytes([c]))
    for c in UPPER:
        pool["cap"][1].append(bytes([c]))
    for c in PUNCT:
        pool["punct"][1].append(bytes([c]))
    pool["space_lower"][1].append(b" ")
    pool["space_cap"][1].append(b" ")
    for c in range(0x80, 0x100):
        pool["high"][1].append(bytes([c]))
    counts = _length_counts()

    def add(t, cat):
        if t in have:
            return False
        have.add(t)
        toks.append(t)
        pool[cat][len(t)].append(t)
        return True

    def pick(cat, L):
        lst = pool[cat].get(L)
        if not lst:
            return None
        return lst[int(len(lst) * rng.random() ** 2.5)]

    def concat(cat_a, cat_b, L):
        k = int(rng.integers(1, L))
        a, b = pick(cat_a, k), pick(cat_b, L - k)
        if a is None or b is None:
            return None
        return a + b

    runs = {b"-": 128, b"=": 32, b"#": 16, b"*": 16, b"_": 16, b"/": 8, b" ": 16}
    for L in range(2, 129):
        n_L = counts[L]
        made = 0
        # fixed families: runs of one character, newline + indentation, digits
        fixed = []
        for ch, maxlen in runs.items():
            if L <= maxlen:
                fixed.append((ch * L, "space" if ch == b" " else "punct"))
        if L <= 17:
            fixed.append((b"\n" + b" " * (L - 1), "nl"))
        if L <= 6:
            fixed.append((b"\n" * L, "nl"))
            fixed.append((b"\n" + b"\t" * (L - 1), "nl"))
        if L == 2:
            fixed += [(bytes([a, b]), "digit") for a in b"0123456789" for b in b"0123456789"]
        if L == 3:
            fixed += [(bytes([a, b, c]), "digit") for a in b"0123456789" for b in b"0123456789"
                      for c in b"0123456789"]
        for t, cat in fixed:
            if made < n_L and add(t, cat):
                made += 1
        # punctuation and high-byte pieces
        quota = {"punct": {2: 300, 3: 400, 4: 300}.get(L, 100 if L <= 8 else 0),
                 "high": {2: n_L - made - 1300 - 300, 3: 800, 4: 300}.get(L, 0)}
        for cat in ("punct", "high"):
            want, tries = quota[cat], 0
            while want > 0 and made < n_L and tries < 50 * quota[cat] + 100:
                tries += 1
                if cat == "high" and L == 2:
                    t = bytes([int(rng.integers(0xC2, 0xF0)), int(rng.integers(0x80, 0xC0))])
                else:
                    t = concat(cat, cat, L)
                if t is not None and add(t, cat):
                    made += 1
                    want -= 1
        # letters: lower, " lower", Cap, " Cap"
        forms = [("lower", "lower", "lower", 0.40), ("space_lower", "lower", "space_lower", 0.42),
                 ("cap", "lower", "cap", 0.08), ("space_cap", "lower", "space_cap", 0.10)]
        probs = np.array([f[3] for f in forms])
        tries = 0
        while made < n_L:
            tries += 1
            if tries > 200 * n_L + 10000:
                raise RuntimeError(f"table generator stuck at length {L}")
            ca, cb, cat, _ = forms[int(rng.choice(4, p=probs))]
            if cat == "space_cap" and L == 2:
                t = b" " + pick("cap", 1)
            else:
                t = concat(ca, cb, L)
            if t is not None and add(t, cat):
                made += 1
    assert len(toks) == 100256, len(toks)
    return toks


def letter_words(table):
    """Tokens of two or more ASCII letters, in rank order (the prose vocabulary)."""
    return [t for t in table if len(t) >= 2 and t.isalpha() and t.isascii()]


def prose_text(table, n_bytes, seed=None, rng=None, zipf_s=1.05):
    """Prose: Zipf(s) draws over the table's letter tokens, single spaces,
    the tiny workload's punctuation / digit / newline mix."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    words = letter_words(table)
    return _slot_text(rng, words, _zipf_cdf(len(words), zipf_s), n_bytes)


# --------------------------------------------------------------------------
# JSON, code and white-space blocks (agentic prompt and tool outputs).

def _hex(rng, n):
    return bytes(np.frombuffer(b"0123456789abcdef", np.uint8)[rng.integers(0, 16, size=n)])


def _json_value(rng, words, cdf, depth, out, indent, level):
    r = rng.random()
    if depth > 0 and r < 0.25:
        n = int(rng.integers(1, 6))
        out.append(b"{")
        for i in range(n):
            if indent:
                out.append(b"\n" + b" " * (indent * (level + 1)))
            out.append(b'"' + words[_zipf_draw(rng, cdf, 1)[0]] + b'":')
            if indent or rng.random() < 0.5:
                out.append(b" ")
            _json_value(rng, words, cdf, depth - 1, out, indent, level + 1)
            if i + 1 < n:
                out.append(b",")
        if indent:
            out.append(b"\n" + b" " * (indent * level))
        out.append(b"}")
    elif depth > 0 and r < 0.35:
        n = int(rng.integers(1, 5))
        out.append(b"[")
        for i in range(n):
            _json_value(rng, words, cdf, depth - 1, out, indent, level + 1)
            if i + 1 < n:
                out.append(b", ")
        out.append(b"]")
    elif r < 0.55:
        out.append(str(int(rng.integers(0, 10 ** int(rng.integers(1, 10))))).encode())
    elif r < 0.62:
        out.append(f"{rng.normal() * 1000:.{int(rng.integers(1, 6))}f}".encode())
    elif r < 0.72:
        out.append(b'"' + _hex(rng, int(rng.choice([8, 16, 32, 40]))) + b'"')
    elif r < 0.76:
        out.append([b"true", b"false", b"null"][int(rng.integers(0, 3))])
    else:
        n = int(rng.integers(1, 6))
        ws = [words[i] for i in _zipf_draw(rng, cdf, n)]
        out.append(b'"' + b" ".join(ws) + b'"')


def json_text(words, cdf, n_bytes, rng):
    out, size = [], 0
    while size < n_bytes:
        part = []
        indent = int(rng.choice([0, 2, 4]))
        _json_value(rng, words, cdf, 3, part, indent, 0)
        part.append(b"\n")
        p = b"".join(part)
        out.append(p)
        size += len(p)
    return b"".join(out)[:n_bytes]


_OPS = [b" = ", b" + ", b" - ", b" * ", b" == ", b" != ", b" && ", b" || ", b" -> ", b".", b", "]


def code_text(words, cdf, n_bytes, rng):
    out, size, level = [], 0, 0
    while size < n_bytes:
        r = rng.random()
        ind = b"\t" * level if rng.random() < 0.15 else b" " * (4 * level)
        w = [words[i] for i in _zipf_draw(rng, cdf, 4)]
        if r < 0.2 and level < 5:
            line = ind + b"def " + w[0] + b"_" + w[1] + b"(" + w[2] + b", " + w[3] + b"):"
            level += 1
        elif r < 0.3 and level < 5:
            line = ind + b"if (" + w[0] + _OPS[int(rng.integers(0, 11))] + w[1] + b") {"
            level += 1
        elif r < 0.45 and level > 0:
            level -= 1
            line = (b"\t" * level if rng.random() < 0.15 else b" " * (4 * level)) + b"}"
        elif r < 0.55:
            line = ind + b"// " + b" ".join(w)
        elif r < 0.65:
            line = b""
        else:
            line = (ind + w[0] + _OPS[int(rng.integers(0, 11))] + w[1] + b"(" +
                    str(int(rng.integers(0, 1000))).encode() + b', "' + w[2] + b'");')
        line += b"\n"
        out.append(line)
        size += len(line)
    return b"".join(out)[:n_bytes]


def ws_run(rng, n, pure):
    if pure:
        return b" " * n
    a = np.full(n, 0x20, np.uint8)
    k = max(1, n // 200)
    pos = rng.integers(0, n, size=k)
    a[pos] = np.where(rng.random(k) < 0.6, 0x0A, 0x09).astype(np.uint8)
    return a.tobytes()


# --------------------------------------------------------------------------
# Agentic prompt: 2,000 typed segments, alternating allow_special true/false.

_ROLES = [b"user", b"assistant", b"tool", b"system"]


def _mixed_block(rng, table_words, cdf, n_bytes, kind):
    if kind == 0:
        return _slot_text(rng, table_words, cdf, n_bytes)
    if kind == 1:
        return json_text(table_words, cdf, n_bytes, rng)
    return code_text(table_words, cdf, n_bytes, rng)


def agentic_segments(table, seed=3, scale=1.0):
    """~4 M characters in 2,000 segments, starting with an allow_special one.

    False segments mix prose 40% / JSON 30% / code 20% / white-space runs 10%
    (run lengths log-uniform in [1, 60,000]; one run of exactly 60,000, one
    straddling character 400,000 of the longest segment). Three false
    segments exceed 400,000 characters (the longest about 1.2 M). About 1% of
    false segments embed literal special strings. `scale` shrinks every length
    for small parity cases."""
    rng = np.random.default_rng(seed)
    words = letter_words(table)
    cdf = _zipf_cdf(len(words), 1.05)
    specials = [s.encode() for s in SPECIALS]
    n_false = 1000
    big = [int(1_200_000 * scale), int(450_000 * scale), int(420_000 * scale)]
    rest_total = int(4_000_000 * scale) - sum(big)
    ln = rng.lognormal(mean=np.log(1200.0), sigma=1.2, size=n_false - 3)
    small = np.maximum(1, (ln / ln.sum() * rest_total).astype(np.int64))
    lengths = big + [int(x) for x in small]
    order = rng.permutation(n_false)
    lengths = [lengths[i] for i in order]
    big_pos = [int(np.where(order == k)[0][0]) for k in range(3)]
    embed = set(int(i) for i in rng.choice(n_false, size=10, replace=False))
    segs = []
    for f in range(n_false):
        k = int(rng.integers(1, 4))
        sp = [specials[int(rng.integers(0, len(specials)))] for _ in range(k)]
        if rng.random() < 0.10:
            sp.insert(1, _ROLES[int(rng.integers(0, 4))])
        segs.append((b"".join(sp), True))
        L = lengths[f]
        parts, size = [], 0
        forced = []
        if f == big_pos[0]:
            forced = [(int(380_000 * scale), 60_000 if scale >= 1 else max(1, int(60_000 * scale)), True),
                      (int(395_000 * scale), int(30_000 * scale) or 1, False)]
        elif f in big_pos[1:]:
            forced = [(int(100_000 * scale), int(28_000 * scale) or 1, True)]
        fi = 0
        while size < L:
            if fi < len(forced) and size >= forced[fi][0]:
                _, n, pure = forced[fi]
                blk = ws_run(rng, min(n, L - size), pure)
                fi += 1
            else:
                kind = int(rng.choice(4, p=[0.40 / 0.9 * 0.9, 0.30, 0.20, 0.10]))
                if kind == 3:
                    n = int(np.exp(rng.uniform(0, np.log(60_000 * max(scale, 1e-3)))))
                    blk = ws_run(rng, max(1, min(n, L - size)), rng.random() < 0.7)
                else:
                    n = int(rng.integers(200, 3000))
                    blk = _mixed_block(rng, words, cdf, min(n, L - size), kind)
            parts.append(blk)
            size += len(blk)
        text = b"".join(parts)[:L]
        if f in embed and len(text) > 40:
            pos = int(rng.integers(0, len(text) - 20))
            text = text[:pos] + specials[int(rng.integers(0, len(specials)))] + text[pos:]
        segs.append((text, False))
    return segs


# --------------------------------------------------------------------------
# Multilingual stress: a 20,000-merge extension over UTF-8 sequences, and
# 8 MiB of ASCII / CJK / Devanagari / emoji / control bytes.

_CJK_COMMON = None


def _cjk_chars(rng):
    return [chr(c) for c in rng.choice(np.arange(0x4E00, 0xA000), size=3000, replace=False)]


def _cjk_block(rng, chars, cdf, n_bytes):
    out, size = [], 0
    while size < n_bytes:
        k = int(rng.integers(5, 31))
        s = "".join(chars[i] for i in _zipf_draw(rng, cdf, k)) + ("，" if rng.random() < 0.6 else "。")
        b = s.encode()
        out.append(b)
        size += len(b)
    return b"".join(out)


def _deva_block(rng, n_bytes):
    cons = [chr(c) for c in range(0x0915, 0x093A)]
    matra = [chr(c) for c in range(0x093E, 0x094D)]
    out, size = [], 0
    while size < n_bytes:
        w = []
        for _ in range(int(rng.integers(1, 5))):
            w.append(cons[int(rng.integers(0, len(cons)))])
            r = rng.random()
            if r < 0.5:
                w.append(matra[int(rng.integers(0, len(matra)))])
            elif r < 0.6:
                w.append("्")
        s = "".join(w) + ("। " if rng.random() < 0.1 else " ")
        b = s.encode()
        out.append(b)
        size += len(b)
    return b"".join(out)


def _emoji_block(rng, n_bytes):
    out, size = [], 0
    while size < n_bytes:
        k = int(rng.integers(1, 5))
        s = "".join(chr(int(c)) for c in rng.integers(0x1F300, 0x1FB00, size=k)) + " "
        b = s.encode()
        out.append(b)
        size += len(b)
    return b"".join(out)


_CTRL = bytes(list(range(0x00, 0x09)) + list(range(0x0E, 0x20)) + [0x7F])


def _ctrl_block(rng, words, cdf, n_bytes):
    out, size = [], 0
    while size < n_bytes:
        k = int(rng.integers(1, 9))
        b = bytes(np.frombuffer(_CTRL, np.uint8)[rng.integers(0, len(_CTRL), size=k)])
        b += b" " + words[_zipf_draw(rng, cdf, 1)[0]] + b" "
        out.append(b)
        size += len(b)
    return b"".join(out)


def multilingual_text(table, n_bytes=8 * MiB, seed=4):
    """Alternating blocks by byte share: ASCII prose 35%, CJK 30% (，/。 every
    5-30 characters), Devanagari 20%, emoji 10%, control bytes 5% (with NUL)."""
    rng = np.random.default_rng(seed)
    words = letter_words(table)
    wcdf = _zipf_cdf(len(words), 1.05)
    chars = _cjk_chars(np.random.default_rng(seed + 1000))
    ccdf = _zipf_cdf(len(chars), 1.1)
    shares = [0.35, 0.30, 0.20, 0.10, 0.05]
    out, size = [], 0
    while size < n_bytes:
        kind = int(rng.choice(5, p=shares))
        n = int(rng.integers(500, 5000))
        if kind == 0:
            blk = _slot_text(rng, words, wcdf, n)
        elif kind == 1:
            blk = _cjk_block(rng, chars, ccdf, n)
        elif kind == 2:
            blk = _deva_block(rng, n)
        elif kind == 3:
            blk = _emoji_block(rng, n)
        else:
            blk = _ctrl_block(rng, words, wcdf, n)
        out.append(blk)
        size += len(blk)
    text = b"".join(out)
    # cut at a character boundary at or below n_bytes
    cut = n_bytes
    while cut > 0 and (text[cut] & 0xC0) == 0x80:
        cut -= 1
    return text[:cut]


def multilingual_table(table, seed=4, n_new=20000):
    """(token bytes, id) pairs for ids 100,277 .. 100,276 + n_new: each new token
    is the concatenation of two existing tokens, at least one of them
    non-ASCII, taken from byte windows of CJK / Devanagari / emoji text
    (whole characters and mid-character fragments)."""
    rng = np.random.default_rng(seed + 7)
    chars = _cjk_chars(np.random.default_rng(seed + 1000))
    ccdf = _zipf_cdf(len(chars), 1.1)
    sample = (_cjk_block(rng, chars, ccdf, 300_000) + _deva_block(rng, 200_000) +
              _emoji_block(rng, 100_000))
    have = set(table)
    new = []
    quota = {2: 1500, 3: 6000, 4: 2500, 5: 1500, 6: 3500, 7: 1200, 8: 1000, 9: 1200,
             10: 600, 11: 400, 12: 600}
    assert sum(quota.values()) == n_new
    arr = np.frombuffer(sample, np.uint8)
    for L in range(2, 13):
        want, tries = quota[L], 0
        while want > 0:
            tries += 1
            if tries > 400 * quota[L]:
                raise RuntimeError(f"multilingual table stuck at length {L}")
            p = int(rng.integers(0, len(arr) - L))
            w = arr[p:p + L].tobytes()
            if w in have or max(w) < 0x80:
                continue
            ks = [k for k in range(1, L) if w[:k] in have and w[k:] in have]
            if not ks:
                continue
            have.add(w)
            new.append(w)
            want -= 1
    return [(t, 100277 + i) for i, t in enumerate(new)]


# --------------------------------------------------------------------------
# Serving batch: 4,096 requests, 256 MiB, heavy reuse.

def _fresh_pool(table, n_bytes, rng):
    """Tool-output text: prose, JSON and hex hashes."""
    words = letter_words(table)
    cdf = _zipf_cdf(len(words), 1.05)
    out, size = [], 0
    while size < n_bytes:
        r = rng.random()
        n = int(rng.integers(2000, 20000))
        if r < 0.6:
            blk = _slot_text(rng, words, cdf, n)
        elif r < 0.9:
            blk = json_text(words, cdf, n, rng)
        else:
            blk = b"\n".join(b"sha256:" + _hex(rng, 64) for _ in range(n // 72 + 1))
        out.append(blk)
        size += len(blk)
    return np.frombuffer(b"".join(out)[:n_bytes], np.uint8)


def serving_batch(table, seed=5, total=256 * MiB, n_req=4096, sigma=2.797, median=8192,
                  max_len=400_000):
    """Returns (text uint8[total], seg_off int64[n_req+1]).

    Lengths: log-normal (median 8,192, sigma 2.797), clipped at 400,000, the
    tail rescaled so the lengths sum to `total`. Request 0 is fresh; request
    i > 0 repeats a request drawn uniformly from the previous 64 (cyclically
    if shorter) for its first 90% and ends in a fresh tool-output suffix."""
    rng = np.random.default_rng(seed)
    L = np.minimum(rng.lognormal(np.log(median), sigma, size=n_req), max_len)
    L = np.maximum(L, 1).astype(np.int64)
    diff = total - int(L.sum())
    i = n_req - 1
    while diff != 0 and i >= 0:
        new = int(min(max_len, max(1, L[i] + diff)))
        diff -= new - int(L[i])
        L[i] = new
        i -= 1
    assert int(L.sum()) == total, (int(L.sum()), total)
    fresh_need = int(L[0]) + int(sum(int(x) - int(0.9 * x) for x in L[1:]))
    pool = _fresh_pool(table, fresh_need + 1, rng)
    text = np.empty(total, np.uint8)
    off = np.zeros(n_req + 1, np.int64)
    np.cumsum(L, out=off[1:])
    fp = 0
    for r in range(n_req):
        a, n = int(off[r]), int(L[r])
        if r == 0:
            text[a:a + n] = pool[fp:fp + n]
            fp += n
            continue
        rep = int(0.9 * n)
        j = int(rng.integers(max(0, r - 64), r))
        src = text[off[j]:off[j + 1]]
        if rep:
            text[a:a + rep] = np.resize(src, rep)
        k = n - rep
        text[a + rep:a + n] = pool[fp:fp + k]
        fp += k
    return text, off


# --------------------------------------------------------------------------

def pack_segments(segments):
    """[(bytes, allow)] -> (text uint8, seg_off int64[S+1], allow uint8[S])."""
    parts = [s for s, _ in segments]
    text = np.frombuffer(b"".join(parts), np.uint8) if parts else np.zeros(0, np.uint8)
    off = np.zeros(len(parts) + 1, np.int64)
    if parts:
        np.cumsum([len(p) for p in parts], out=off[1:])
    allow = np.asarray([1 if a else 0 for _, a in segments], np.uint8)
    return text, off, allow


def input_sha256(text, seg_off, allow):
    """sha256 of one workload input: its text, segment offsets (int64) and
    allow_special flags (uint8), in that order, as raw bytes."""
    import hashlib
    h = hashlib.sha256()
    for a in (np.ascontiguousarray(text, np.uint8), np.ascontiguousarray(seg_off, np.int64),
              np.ascontiguousarray(allow, np.uint8)):
        h.update(a.tobytes())
    return h.hexdigest()


def table_sha256(ranks):
    """sha256 of a rank table: for each token in rank order its id (int64) and
    its length (int64), then the token's bytes."""
    import hashlib
    h = hashlib.sha256()
    for i, t in enumerate(ranks):
        tok, tid = (t if isinstance(t, tuple) else (t, i))
        h.update(np.array([tid, len(tok)], np.int64).tobytes())
        h.update(tok)
    return h.hexdigest()


def manifest_inputs(serving_total=256 * MiB):
    """The inputs the manifest records: name -> (text, seg_off, allow)."""
    table = full_table()
    tiny = np.frombuffer(tiny_input(), np.uint8)
    prose = np.frombuffer(prose_text(table, 1 * MiB, seed=2), np.uint8)
    one = lambda t: (t, np.array([0, t.size], np.int64), np.zeros(1, np.uint8))  # noqa: E731
    ag = pack_segments(agentic_segments(table, seed=3))
    ml = multilingual_text(table, seed=4)
    ml = np.frombuffer(ml.tobytes() if isinstance(ml, np.ndarray) else bytes(ml), np.uint8)
    out = {"tiny": one(tiny), "prose": one(prose), "agentic": ag, "multilingual": one(ml)}
    if serving_total:
        text, off = serving_batch(table, seed=5, total=serving_total)
        out["serving"] = (text, off, np.zeros(len(off) - 1, np.uint8))
    return out
