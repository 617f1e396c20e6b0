"""Independent pins for the oracle (test helpers; no oracle code here).

- regex_split: the printed cl100k split pattern run by the `regex` library
  (possessive quantifiers and \\p{..} classes), an independent matcher.
- naive_bpe: brute force merge that rebuilds the piece list and rescans every
  adjacent pair at every step (no incremental bookkeeping).
- closed_form_cuts: the 25k-run chunking rule in closed form (cut at run start
  + 25,000*k), against the oracle's character-by-character loop.
"""
# The pattern as printed in "tiktoken Deep Dive", "The split pattern" (its five
# printed lines joined as one alternation).
SPLIT_PATTERN = (r"""'(?i:[sdmt]|ll|ve|re)|[^\r\n\p{L}\p{N}]?+\p{L}++|\p{N}{1,3}+"""
                 r"""| ?[^\s\p{L}\p{N}]++[\r\n]*+|\s++$|\s*[\r\n]|\s+(?!\S)|\s""")

# The same alternation with r50k's digit clause in place of cl100k's ("tiktoken
# Deep Dive", "r50k, cl100k, o200k": r50k used " ?\p{N}++", an unbounded digit
# run with an optional leading space).
SPLIT_PATTERN_R50K_DIGITS = SPLIT_PATTERN.replace(r"\p{N}{1,3}+", r" ?\p{N}++")
assert SPLIT_PATTERN_R50K_DIGITS != SPLIT_PATTERN

_compiled = {}


def regex_split(text, pattern=SPLIT_PATTERN):
    import regex
    if pattern not in _compiled:
        _compiled[pattern] = regex.compile(pattern)
    s = text.decode("utf-8") if isinstance(text, bytes) else text
    return [m.group(0).encode("utf-8") for m in _compiled[pattern].finditer(s)]


def naive_bpe(piece, ranks):
    """ranks: dict bytes -> rank. Merge the leftmost lowest-ranked adjacent pair
    until no adjacent pair is a token; returns the list of ranks."""
    parts = [piece[i:i + 1] for i in range(len(piece))]
    while True:
        best, best_i = None, -1
        for i in range(len(parts) - 1):
            r = ranks.get(parts[i] + parts[i + 1])
            if r is not None and (best is None or r < best):
                best, best_i = r, i
        if best is None:
            break
        parts = parts[:best_i] + [parts[best_i] + parts[best_i + 1]] + parts[best_i + 2:]
    return [ranks[p] for p in parts]


def closed_form_cuts(is_space, window=400_000, run=25_000):
    """Chunk starts (character indices) of one segment: windows of `window`
    characters; inside each window every maximal run of equal space-ness that
    starts at r is cut at r + run*k (k >= 1) strictly inside the run."""
    n = len(is_space)
    cuts = []
    for w in range(0, n, window):
        e = min(n, w + window)
        cuts.append(w)
        r = w
        while r < e:
            q = r
            while q < e and is_space[q] == is_space[r]:
                q += 1
            k = r + run
            while k < q:
                cuts.append(k)
                k += run
            r = q
    return cuts
