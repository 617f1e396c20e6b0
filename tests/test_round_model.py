"""The chunked exact rounds of the big-piece merge, as a CPU model.

The CTA merge of 1,025-32,768-byte pre-tokens keeps the piece's parts in
warp-owned chunks: each chunk holds a run of parts in text order at the front
of its window, and a part's pair rank is the rank with the next part in text
order (the first part of the next non-empty chunk for a chunk's last part).
A round takes the minimum pair rank rs, chooses every other rs-pair from the
start of each run of rs-pairs (a run that enters a chunk from the chunks
before it flips the chunk's leading choices when its length there is odd),
stops after the first chosen merge that creates a neighbour pair ranked below
rs, and compacts every chunk in place.  A round whose rank cannot stop early
takes a chunk's entering run and whether its first part is taken from the
counts of rs-pairs that lead and end each chunk.

This model restates those steps in Python and checks them against the plain
parts loop (merge the leftmost lowest-ranked adjacent pair until none is left;
"tiktoken Deep Dive", "Inside encode") on random small tables, including
tables whose ranks are shuffled so that the stop rule fires, with 1-16 chunks
of every size down to one part and empty ones.
"""
import random

INF = 1 << 30


def parts_loop(ids, pr):
    parts = list(ids)
    while True:
        best, at = INF, -1
        for i in range(len(parts) - 1):
            r = pr(parts[i], parts[i + 1])
            if r < best:
                best, at = r, i
        if at < 0:
            return parts
        parts[at:at + 2] = [best]


def chunked_rounds(ids, pr, nw, cw, flip=True):
    """The chunked rounds over nw chunks of cw slots; returns (ids, rounds,
    rounds stopped early).  flip=False plants a mistake: the run entering a
    chunk is ignored."""
    ch = [list(ids[w * cw:(w + 1) * cw]) for w in range(nw)]

    def nxt(w, j):
        if j + 1 < len(ch[w]):
            return w, j + 1
        for v in range(w + 1, nw):
            if ch[v]:
                return v, 0
        return None

    def prv(w, j):
        if j > 0:
            return w, j - 1
        for v in range(w - 1, -1, -1):
            if ch[v]:
                return v, len(ch[v]) - 1
        return None

    def ranks():
        out = []
        for w in range(nw):
            row = []
            for j in range(len(ch[w])):
                s = nxt(w, j)
                row.append(pr(ch[w][j], ch[s[0]][s[1]]) if s else INF)
            out.append(row)
        return out

    def stats(rk):
        # per chunk: minimum rank, pairs of it before the first other pair
        # (lead) and after the last other pair (tail)
        mn, lead, tail = [], [], []
        for w in range(nw):
            m = min(rk[w]) if rk[w] else INF
            other = [j for j, r in enumerate(rk[w]) if r != m]
            mn.append(m)
            lead.append(other[0] if other else len(rk[w]))
            tail.append(len(rk[w]) - 1 - (other[-1] if other else -1))
        return mn, lead, tail

    rounds = stopped = 0
    rk = ranks()
    while True:
        mn, lead, tail = stats(rk)
        rs = min(mn)
        if rs == INF:
            break
        rounds += 1
        cnt = [len(c) for c in ch]

        def run_into(v):
            r = 0
            for u in range(v - 1, -1, -1):
                if cnt[u] == 0:
                    continue
                if mn[u] != rs:
                    break
                r += tail[u]
                if lead[u] != cnt[u]:
                    break
            return r

        # choices, counting the run that enters each chunk
        sel = []
        for w in range(nw):
            row = [False] * cnt[w]
            if mn[w] == rs:
                last_other = -1 - (run_into(w) if flip and lead[w] > 0 else 0)
                for j in range(cnt[w]):
                    if rk[w][j] != rs:
                        last_other = j
                    else:
                        row[j] = (j - last_other - 1) % 2 == 0
            sel.append(row)
        # the first chosen merge (text order) that creates a lower-ranked pair
        limit = (nw, 0)
        for w in range(nw):
            for j in range(cnt[w]):
                if not sel[w][j]:
                    continue
                p = prv(w, j)
                bad = False
                if p is not None:
                    pp = prv(*p)
                    left = rs if (pp is not None and sel[pp[0]][pp[1]]) else ch[p[0]][p[1]]
                    bad = pr(left, rs) < rs
                s = nxt(w, j)
                ss = nxt(*s) if s else None
                if ss is not None and pr(rs, ch[ss[0]][ss[1]]) < rs:
                    bad = True
                if bad:
                    limit = min(limit, (w, j))
        # in a round that does not stop early, a chunk's first part is taken
        # exactly when the last pair before it is an rs-pair at an even place
        # in its run (what the one-pass round computes from the counts alone)
        stopped += limit != (nw, 0)
        if limit == (nw, 0) and flip:
            for w in range(nw):
                if cnt[w] == 0:
                    continue
                v = w - 1
                while v >= 0 and cnt[v] == 0:
                    v -= 1
                gone = False
                if v >= 0 and mn[v] == rs and tail[v] > 0:
                    at = (run_into(v) if lead[v] == cnt[v] else 0) + tail[v] - 1
                    gone = at % 2 == 0
                assert gone == (v >= 0 and sel[v][-1])
        # merge and compact in place
        new = []
        for w in range(nw):
            keep = []
            for j in range(cnt[w]):
                p = prv(w, j)
                if p is not None and sel[p[0]][p[1]] and p <= limit:
                    continue
                keep.append(rs if sel[w][j] and (w, j) <= limit else ch[w][j])
            new.append(keep)
        ch = new
        rk = ranks()
    return [t for c in ch for t in c], rounds, stopped


def make_table(rng, alpha, n_new, shuffle):
    toks = [bytes([c]) for c in alpha]
    seen = set(toks)
    for _ in range(n_new):
        t = rng.choice(toks) + rng.choice(toks)
        if t not in seen and len(t) <= 12:
            seen.add(t)
            toks.append(t)
    if shuffle:
        head, tail = toks[:len(alpha)], toks[len(alpha):]
        rng.shuffle(tail)
        toks = head + tail
    return toks, {t: i for i, t in enumerate(toks)}


def _trials(seed, count):
    rng = random.Random(seed)
    for trial in range(count):
        alpha = (b"ab", b"abc", b"a b\t")[trial % 3]
        toks, rank = make_table(rng, alpha, rng.randint(3, 40), shuffle=trial % 2 == 1)

        def pr(x, y, toks=toks, rank=rank):
            return rank.get(toks[x] + toks[y], INF)

        n = rng.randint(1, 70)
        ids = [rank[bytes([rng.choice(alpha)])] for _ in range(n)]
        nw = rng.choice([1, 2, 3, 4, 8, 16])
        cw = rng.choice([1, 2, 3, 5, 8])
        if cw * nw < n:
            cw = -(-n // nw)
        yield ids, pr, nw, cw


def test_chunked_rounds_equal_the_parts_loop():
    stopped = 0
    for ids, pr, nw, cw in _trials(17, 2500):
        got, _, st = chunked_rounds(ids, pr, nw, cw)
        assert got == parts_loop(ids, pr), (ids, nw, cw)
        stopped += st
    assert stopped > 100  # the shuffled tables exercise the stop rule


def test_model_catches_a_dropped_flip():
    """Planted mistake: the run of rs-pairs entering a chunk is ignored."""
    wrong = sum(chunked_rounds(ids, pr, nw, cw, flip=False)[0] != parts_loop(ids, pr)
                for ids, pr, nw, cw in _trials(19, 600))
    assert wrong > 0
