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


def naive_train(corpus, n_merges):
    """Brute-force BPE trainer: split the corpus with the printed pattern (the
    regex library), count identical pre-tokens, then n_merges times recount
    every adjacent pair of every word from scratch, take the most frequent pair
    whose concatenation is not a token yet (ties: the smallest (left id, right
    id)), add it as the next id and join its occurrences left to right.
    Returns the learned token byte strings in id order."""
    from collections import Counter
    words = Counter(regex_split(corpus))
    seqs = [([w[i:i + 1] for i in range(len(w))], c) for w, c in words.items()]
    ids = {bytes([b]): b for b in range(256)}
    learned = []
    for _ in range(n_merges):
        counts = Counter()
        for parts, c in seqs:
            for a, b in zip(parts, parts[1:]):
                counts[(a, b)] += c
        best = None
        for (a, b), c in counts.items():
            if a + b in ids:
                continue
            key = (-c, ids[a], ids[b])
            if best is None or key < best[0]:
                best = (key, a, b)
        if best is None:
            break
        _, a, b = best
        ids[a + b] = 256 + len(learned)
        learned.append(a + b)
        for k, (parts, c) in enumerate(seqs):
            out, i = [], 0
            while i < len(parts):
                if i + 1 < len(parts) and parts[i] == a and parts[i + 1] == b:
                    out.append(a + b)
                    i += 2
                else:
                    out.append(parts[i])
                    i += 1
            seqs[k] = (out, c)
    return learned
