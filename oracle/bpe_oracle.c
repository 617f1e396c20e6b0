/*
 * bpe_oracle.c -- plain, single-threaded CPU oracle for byte-level BPE encoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  It shares
 * no code, header, table or generator with the CUDA path, and it is written to
 * be checked by eye against the pages it follows, not to be fast:
 *
 *   [TT]  "tiktoken Deep Dive": "An encoding is three objects", "The byte floor",
 *         "The split pattern", "Inside encode: a parts vector and a linear scan",
 *         "Special tokens and the injection nobody plans for".
 *   [BT]  "Making Kimi K3 Tokenization 18x Faster For Million Token Agentic
 *         Workloads": "Why Kimi K3 tokenization is non-trivial" (typed
 *         segments) and "One native call for the whole serving path" (the
 *         400k-character / 25k-character safe chunking).
 *
 * Readings taken where the pages are silent or garbled (each also listed in
 * the design notes):
 *   - the printed split pattern is one alternation, tried in printed order;
 *   - `$` is the end of the ordinary text piece being split;
 *   - argmin ties in the parts loop go to the leftmost pair;
 *   - the parts vector's last two entries hold the MAX sentinel;
 *   - safe chunking counts code points, runs of Python-`isspace` characters,
 *     and comes before special matching (a special cut by a chunk boundary is
 *     ordinary text);
 *   - specials: leftmost match, longest special at that position;
 *   - allow_special = 0 encodes literal special strings as ordinary text.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "unicode_ranges.h"

#define ORC_OK 0
#define ORC_E_ARG (-1)
#define ORC_E_TABLE (-2)
#define ORC_E_UTF8 (-3)
#define ORC_E_CAPACITY (-4)
#define ORC_E_NOMEM (-6)
#define ORC_E_BADID (-8)

#define ORC_PATTERN_CL100K 1      /* the pattern printed on the tiktoken page */
#define ORC_PATTERN_R50K_DIGITS 2 /* the same with r50k's digit clause */

#define RANK_MAX 0xFFFFFFFFu
#define CHUNK_CHARS 400000   /* [BT] "at most 400k characters" */
#define RUN_CHARS 25000      /* [BT] "runs ... at 25k characters" */

/* ------------------------------------------------------------------------- */
/* Unicode classes ([TT] "The split pattern": \p{L}, \p{N}, \s).              */

enum { CLS_OTHER = 0, CLS_L = 1, CLS_N = 2, CLS_WS = 3 };

static int cp_class(uint32_t c) {
  int lo = 0, hi = ORC_NRANGES - 1;
  while (lo <= hi) {
    int mid = (lo + hi) / 2;
    if (c < ORC_RANGES[mid][0]) hi = mid - 1;
    else if (c > ORC_RANGES[mid][1]) lo = mid + 1;
    else return (int)ORC_RANGES[mid][2];
  }
  return CLS_OTHER;
}
static int is_L(uint32_t c) { return cp_class(c) == CLS_L; }
static int is_N(uint32_t c) { return cp_class(c) == CLS_N; }
static int is_WS(uint32_t c) { return cp_class(c) == CLS_WS; }
static int is_CRLF(uint32_t c) { return c == 0x0A || c == 0x0D; }
/* [^\s\p{L}\p{N}] */
static int is_other(uint32_t c) { return cp_class(c) == CLS_OTHER; }
/* Python str.isspace(): the white-space test of the legacy chunking rule. */
static int py_isspace(uint32_t c) { return is_WS(c) || (c >= 0x1C && c <= 0x1F); }

int orc_cp_class(uint32_t c) { return cp_class(c); }
int orc_py_isspace(uint32_t c) { return py_isspace(c); }

/* ------------------------------------------------------------------------- */
/* UTF-8 decoding: byte string -> code points, with the byte offset of each.  */

static int utf8_decode(const uint8_t* s, int64_t n, uint32_t* cps, int64_t* boff,
                       int64_t* ncp_out, int64_t* bad_pos) {
  int64_t i = 0, k = 0;
  while (i < n) {
    uint8_t b = s[i];
    uint32_t c;
    int len;
    if (b < 0x80) { c = b; len = 1; }
    else if (b >= 0xC2 && b <= 0xDF) { c = b & 0x1F; len = 2; }
    else if (b >= 0xE0 && b <= 0xEF) { c = b & 0x0F; len = 3; }
    else if (b >= 0xF0 && b <= 0xF4) { c = b & 0x07; len = 4; }
    else { *bad_pos = i; return ORC_E_UTF8; }
    if (i + len > n) { *bad_pos = i; return ORC_E_UTF8; }
    for (int j = 1; j < len; j++) {
      uint8_t t = s[i + j];
      if ((t & 0xC0) != 0x80) { *bad_pos = i; return ORC_E_UTF8; }
      c = (c << 6) | (t & 0x3F);
    }
    /* reject overlong forms, surrogates and values above U+10FFFF */
    if ((len == 3 && c < 0x800) || (len == 4 && c < 0x10000) || c > 0x10FFFF ||
        (c >= 0xD800 && c <= 0xDFFF)) {
      *bad_pos = i;
      return ORC_E_UTF8;
    }
    cps[k] = c;
    boff[k] = i;
    k++;
    i += len;
  }
  boff[k] = n;
  *ncp_out = k;
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* The encoding: mergeable ranks (bytes -> rank = id) plus specials            */
/* ([TT] "An encoding is three objects").                                     */

typedef struct {
  const uint8_t* p;
  int64_t len;
  uint32_t rank;
} orc_entry;

typedef struct {
  uint8_t* rank_bytes;
  orc_entry* by_bytes; /* sorted by byte string, for lookups */
  int64_t n;
  int64_t* by_id;      /* id -> index into rank entries (unsorted copy), or -1 */
  orc_entry* plain;    /* entries in input order (for decode) */
  int64_t max_id;
  uint8_t* spec_bytes;
  int64_t* spec_off;
  int32_t* spec_ids;
  int64_t n_spec;
  int pattern;         /* ORC_PATTERN_CL100K or ORC_PATTERN_R50K_DIGITS */
} orc_enc;

static int cmp_bytes(const uint8_t* a, int64_t la, const uint8_t* b, int64_t lb) {
  int64_t m = la < lb ? la : lb;
  int c = m ? memcmp(a, b, (size_t)m) : 0;
  if (c) return c;
  return (la > lb) - (la < lb);
}
static int cmp_entry(const void* x, const void* y) {
  const orc_entry* a = (const orc_entry*)x;
  const orc_entry* b = (const orc_entry*)y;
  return cmp_bytes(a->p, a->len, b->p, b->len);
}

/* rank of a byte string, or RANK_MAX if it is not a mergeable token */
static uint32_t rank_of(const orc_enc* E, const uint8_t* p, int64_t len) {
  int64_t lo = 0, hi = E->n - 1;
  while (lo <= hi) {
    int64_t mid = lo + (hi - lo) / 2;
    int c = cmp_bytes(p, len, E->by_bytes[mid].p, E->by_bytes[mid].len);
    if (c == 0) return E->by_bytes[mid].rank;
    if (c < 0) hi = mid - 1;
    else lo = mid + 1;
  }
  return RANK_MAX;
}

void orc_free(orc_enc* E) {
  if (!E) return;
  free(E->rank_bytes);
  free(E->by_bytes);
  free(E->by_id);
  free(E->plain);
  free(E->spec_bytes);
  free(E->spec_off);
  free(E->spec_ids);
  free(E);
}

/* Builds an encoding.  Rejects tables that break the byte floor ([TT] "The
 * byte floor": all 256 single bytes are tokens), duplicate byte strings,
 * duplicate ids, and specials whose ids collide with ranks. */
int orc_new(const uint8_t* rank_bytes, const int64_t* rank_off, const uint32_t* rank_ids,
            int64_t n, const uint8_t* spec_bytes, const int64_t* spec_off,
            const int32_t* spec_ids, int64_t n_spec, orc_enc** out) {
  *out = NULL;
  if (n <= 0 || !rank_bytes || !rank_off || !rank_ids || n_spec < 0) return ORC_E_ARG;
  orc_enc* E = (orc_enc*)calloc(1, sizeof(orc_enc));
  if (!E) return ORC_E_NOMEM;
  int64_t nb = rank_off[n];
  E->rank_bytes = (uint8_t*)malloc((size_t)(nb ? nb : 1));
  E->by_bytes = (orc_entry*)malloc(sizeof(orc_entry) * (size_t)n);
  E->plain = (orc_entry*)malloc(sizeof(orc_entry) * (size_t)n);
  if (!E->rank_bytes || !E->by_bytes || !E->plain) { orc_free(E); return ORC_E_NOMEM; }
  memcpy(E->rank_bytes, rank_bytes, (size_t)nb);
  E->n = n;
  E->max_id = -1;
  E->pattern = ORC_PATTERN_CL100K;
  for (int64_t i = 0; i < n; i++) {
    int64_t len = rank_off[i + 1] - rank_off[i];
    if (len <= 0) { orc_free(E); return ORC_E_TABLE; }
    orc_entry e = {E->rank_bytes + rank_off[i], len, rank_ids[i]};
    E->by_bytes[i] = e;
    E->plain[i] = e;
    if ((int64_t)rank_ids[i] > E->max_id) E->max_id = rank_ids[i];
  }
  qsort(E->by_bytes, (size_t)n, sizeof(orc_entry), cmp_entry);
  for (int64_t i = 1; i < n; i++)
    if (cmp_entry(&E->by_bytes[i - 1], &E->by_bytes[i]) == 0) { orc_free(E); return ORC_E_TABLE; }
  for (int b = 0; b < 256; b++) {
    uint8_t byte = (uint8_t)b;
    if (rank_of(E, &byte, 1) == RANK_MAX) { orc_free(E); return ORC_E_TABLE; }
  }
  for (int64_t i = 0; i < n_spec; i++)
    if ((int64_t)spec_ids[i] > E->max_id) E->max_id = spec_ids[i];
  E->by_id = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E->max_id + 1));
  if (!E->by_id) { orc_free(E); return ORC_E_NOMEM; }
  for (int64_t i = 0; i <= E->max_id; i++) E->by_id[i] = -1;
  for (int64_t i = 0; i < n; i++) {
    if (E->by_id[rank_ids[i]] != -1) { orc_free(E); return ORC_E_TABLE; }
    E->by_id[rank_ids[i]] = i;
  }
  E->n_spec = n_spec;
  int64_t sb = n_spec ? spec_off[n_spec] : 0;
  E->spec_bytes = (uint8_t*)malloc((size_t)(sb ? sb : 1));
  E->spec_off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_spec + 1));
  E->spec_ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_spec ? n_spec : 1));
  if (!E->spec_bytes || !E->spec_off || !E->spec_ids) { orc_free(E); return ORC_E_NOMEM; }
  if (sb) memcpy(E->spec_bytes, spec_bytes, (size_t)sb);
  E->spec_off[0] = 0;
  for (int64_t i = 0; i < n_spec; i++) {
    E->spec_off[i + 1] = spec_off[i + 1] - spec_off[0];
    if (spec_off[i + 1] - spec_off[i] <= 0 || spec_ids[i] < 0) { orc_free(E); return ORC_E_TABLE; }
    if (E->by_id[spec_ids[i]] != -1) { orc_free(E); return ORC_E_TABLE; }
    for (int64_t j = 0; j < i; j++)
      if (spec_ids[j] == spec_ids[i]) { orc_free(E); return ORC_E_TABLE; }
    E->spec_ids[i] = spec_ids[i];
  }
  *out = E;
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Byte-pair merge of one pre-token ([TT] "Inside encode: a parts vector and  */
/* a linear scan").  The rule: start from one piece per byte; as long as some */
/* two neighbouring pieces concatenate to a token, join the pair whose token  */
/* has the lowest rank (the leftmost such pair on a tie); then output the     */
/* rank of every piece.  Only the two pairs that touch the joined piece can   */
/* change rank, so only those are looked up again.                            */
/*                                                                            */
/* Pieces are kept as a singly linked list over byte offsets: piece k covers  */
/* bytes [k, nxt[k]) and pr[k] is the rank of piece k joined with the piece   */
/* after it (RANK_MAX when that is not a token or there is no next piece).   */
/* Returns the number of ids written to out (out has room for m ids).         */

int64_t orc_bpe_piece(const orc_enc* E, const uint8_t* b, int64_t m, int32_t* out) {
  if (m <= 0) return 0;
  int64_t* nxt = (int64_t*)malloc(sizeof(int64_t) * (size_t)m);
  uint32_t* pr = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)m);
  if (!nxt || !pr) { free(nxt); free(pr); return -1; }
  for (int64_t k = 0; k < m; k++) {
    nxt[k] = k + 1;
    pr[k] = (k + 1 < m) ? rank_of(E, b + k, 2) : RANK_MAX;
  }
  for (;;) {
    /* walk the pieces left to right: the first piece whose pair rank is the
     * smallest seen so far wins, so ties go to the leftmost pair */
    int64_t win = -1, before = -1, prev = -1;
    uint32_t lo = RANK_MAX;
    for (int64_t k = 0; k < m; k = nxt[k]) {
      if (pr[k] < lo) { lo = pr[k]; win = k; before = prev; }
      prev = k;
    }
    if (win < 0) break; /* no neighbouring pair is a token */
    /* join piece win with its successor */
    nxt[win] = nxt[nxt[win]];
    /* the pair (win, its new successor) and the pair (predecessor, win) */
    pr[win] = (nxt[win] < m) ? rank_of(E, b + win, nxt[nxt[win]] - win) : RANK_MAX;
    if (before >= 0) pr[before] = rank_of(E, b + before, nxt[win] - before);
  }
  int64_t cnt = 0;
  for (int64_t k = 0; k < m; k = nxt[k]) out[cnt++] = (int32_t)rank_of(E, b + k, nxt[k] - k);
  free(nxt);
  free(pr);
  return cnt;
}

/* ------------------------------------------------------------------------- */
/* The split pattern ([TT] "The split pattern"), one clause at a time, tried  */
/* in the printed order at position p of the code points c[0..n) of one       */
/* ordinary text piece.  Returns the length of the match in code points.      */
/*                                                                            */
/*   C1 '(?i:[sdmt]|ll|ve|re)        C5 \s++$                                 */
/*   C2 [^\r\n\p{L}\p{N}]?+\p{L}++   C6 \s*[\r\n]                             */
/*   C3 \p{N}{1,3}+                  C7 \s+(?!\S)                             */
/*   C4  ?[^\s\p{L}\p{N}]++[\r\n]*+  C8 \s                                    */
/*                                                                            */
/* ORC_PATTERN_R50K_DIGITS is the same alternation with r50k's digit clause   */
/* in place of C3 ([TT] "r50k, cl100k, o200k": " ?\p{N}++", an unbounded      */
/* digit run with an optional leading space).                                 */

/* (?i:x) for the ASCII letters of clause 1: simple case folding adds U+017F
 * (LATIN SMALL LETTER LONG S) to s; the other letters fold only to their
 * ASCII pair. */
static int fold_eq(uint32_t c, char x) {
  uint32_t lo = (uint32_t)x, up = (uint32_t)(x - 'a' + 'A');
  if (c == lo || c == up) return 1;
  return x == 's' && c == 0x017F;
}

static int64_t match_clause(const uint32_t* c, int64_t n, int64_t p, int pattern) {
  /* C1: contractions */
  if (c[p] == 0x27 && p + 1 < n) {
    uint32_t a = c[p + 1];
    if (fold_eq(a, 's') || fold_eq(a, 'd') || fold_eq(a, 'm') || fold_eq(a, 't')) return 2;
    if (p + 2 < n) {
      uint32_t b2 = c[p + 2];
      if ((fold_eq(a, 'l') && fold_eq(b2, 'l')) || (fold_eq(a, 'v') && fold_eq(b2, 'e')) ||
          (fold_eq(a, 'r') && fold_eq(b2, 'e')))
        return 3;
    }
  }
  /* C2: one optional (possessive) non-letter/non-number/non-CR/LF prefix, then letters */
  {
    int64_t q = p;
    if (!is_CRLF(c[p]) && !is_L(c[p]) && !is_N(c[p])) q = p + 1;
    if (q < n && is_L(c[q])) {
      while (q < n && is_L(c[q])) q++;
      return q - p;
    }
  }
  if (pattern == ORC_PATTERN_R50K_DIGITS) {
    /* C3 (r50k): an optional space, then every number that follows */
    int64_t q = p;
    if (c[p] == 0x20 && p + 1 < n && is_N(c[p + 1])) q = p + 1;
    if (is_N(c[q])) {
      while (q < n && is_N(c[q])) q++;
      return q - p;
    }
  } else if (is_N(c[p])) {
    /* C3: one to three numbers */
    int64_t q = p;
    while (q < n && q - p < 3 && is_N(c[q])) q++;
    return q - p;
  }
  /* C4: optional space, a run of "other" characters, then CR/LF characters */
  {
    int64_t q = p;
    if (c[p] == 0x20 && p + 1 < n && is_other(c[p + 1])) q = p + 1;
    if (is_other(c[q])) {
      while (q < n && is_other(c[q])) q++;
      while (q < n && is_CRLF(c[q])) q++;
      return q - p;
    }
  }
  if (is_WS(c[p])) {
    int64_t e = p; /* end of the white-space run starting at p */
    int64_t last_crlf = -1;
    while (e < n && is_WS(c[e])) {
      if (is_CRLF(c[e])) last_crlf = e;
      e++;
    }
    /* C5: the run reaches the end of the piece */
    if (e == n) return e - p;
    /* C6: white space up to and including the last CR/LF of the run */
    if (last_crlf >= 0) return last_crlf + 1 - p;
    /* C7: all but the last white-space character (the next one is not \S) */
    if (e - p >= 2) return e - p - 1;
    /* C8: one white-space character */
    return 1;
  }
  return 0; /* unreachable: every code point is L, N, \s or "other" */
}

/* Splits c[0..n) into pre-tokens; writes the start of each (code-point index)
 * to starts[] and returns how many there are. */
int64_t orc_split_cps(const uint32_t* c, int64_t n, int64_t* starts, int pattern) {
  int64_t p = 0, k = 0;
  while (p < n) {
    int64_t len = match_clause(c, n, p, pattern);
    if (len <= 0) return -1;
    starts[k++] = p;
    p += len;
  }
  return k;
}

/* ------------------------------------------------------------------------- */
/* tiktoken-safe chunking ([BT] "One native call for the whole serving        */
/* path"): windows of at most 400,000 characters, then, inside each window,   */
/* a cut before any character that would make the current run of white-space */
/* or non-white-space characters longer than 25,000.  Writes chunk starts     */
/* (code-point indices) and returns how many.                                 */

static int64_t safe_chunks(const uint32_t* c, int64_t n, int64_t* starts) {
  int64_t k = 0;
  for (int64_t w = 0; w < n; w += CHUNK_CHARS) {
    int64_t w_end = w + CHUNK_CHARS < n ? w + CHUNK_CHARS : n;
    starts[k++] = w;
    int cur_space = py_isspace(c[w]);
    int64_t run = 0;
    for (int64_t i = w; i < w_end; i++) {
      int sp = py_isspace(c[i]);
      if (sp != cur_space) {
        cur_space = sp;
        run = 1;
      } else {
        run++;
        if (run > RUN_CHARS) {
          starts[k++] = i;
          run = 1;
        }
      }
    }
  }
  return k;
}

int64_t orc_safe_chunks(const uint32_t* c, int64_t n, int64_t* starts) {
  return safe_chunks(c, n, starts);
}

/* ------------------------------------------------------------------------- */
/* Encoding of segments.                                                      */

typedef struct {
  int32_t* out;
  int64_t cap;
  int64_t count;
  int32_t* scratch; /* room for the ids of one pre-token */
} orc_sink;

static void sink_put(orc_sink* s, int32_t id) {
  if (s->count < s->cap) s->out[s->count] = id;
  s->count++;
}

/* Ordinary text: split with the pattern, then merge each pre-token. */
static int encode_ordinary(const orc_enc* E, const uint8_t* seg, const uint32_t* cps,
                           const int64_t* boff, int64_t c0, int64_t c1, int64_t* starts,
                           orc_sink* sink) {
  int64_t n = c1 - c0;
  if (n <= 0) return ORC_OK;
  int64_t np = orc_split_cps(cps + c0, n, starts, E->pattern);
  if (np < 0) return ORC_E_ARG;
  for (int64_t t = 0; t < np; t++) {
    int64_t a = c0 + starts[t];
    int64_t b = (t + 1 < np) ? c0 + starts[t + 1] : c1;
    int64_t bs = boff[a], be = boff[b];
    int64_t k = orc_bpe_piece(E, seg + bs, be - bs, sink->scratch);
    if (k < 0) return ORC_E_NOMEM;
    for (int64_t j = 0; j < k; j++) sink_put(sink, sink->scratch[j]);
  }
  return ORC_OK;
}

/* One chunk of one segment: the exact-string special pass when specials are
 * allowed ([TT] "Special tokens ..."), ordinary text everywhere else. */
static int encode_chunk(const orc_enc* E, const uint8_t* seg, const uint32_t* cps,
                        const int64_t* boff, int64_t ncp, int64_t c0, int64_t c1, int allow,
                        int64_t* starts, orc_sink* sink) {
  if (!allow || E->n_spec == 0) return encode_ordinary(E, seg, cps, boff, c0, c1, starts, sink);
  int64_t cur = c0; /* first code point not yet emitted */
  int64_t end_b = boff[c1];
  for (int64_t i = c0; i < c1; i++) {
    int64_t pb = boff[i];
    int64_t best = -1, best_len = 0;
    for (int64_t s = 0; s < E->n_spec; s++) {
      int64_t sl = E->spec_off[s + 1] - E->spec_off[s];
      if (pb + sl <= end_b && memcmp(seg + pb, E->spec_bytes + E->spec_off[s], (size_t)sl) == 0 &&
          sl > best_len) {
        best = s;
        best_len = sl;
      }
    }
    if (best < 0) continue;
    int rc = encode_ordinary(E, seg, cps, boff, cur, i, starts, sink);
    if (rc) return rc;
    sink_put(sink, E->spec_ids[best]);
    /* continue after the special (a valid UTF-8 special ends on a character) */
    int64_t j = i;
    while (j < ncp && boff[j] < pb + best_len) j++;
    cur = j;
    i = j - 1;
  }
  return encode_ordinary(E, seg, cps, boff, cur, c1, starts, sink);
}

/* Encodes typed segments ([BT] "Why Kimi K3 tokenization is non-trivial":
 * ordered (text, allow_special) segments, one call).  out_offsets[s] is the
 * index of segment s's first id; out_offsets[S] is the total.  *n_ids always
 * receives the total, even when it exceeds cap (then ORC_E_CAPACITY). */
int orc_encode_segments(const orc_enc* E, const uint8_t* text, const int64_t* seg_off,
                        const uint8_t* allow, int64_t S, int tiktoken_safe, int32_t* out,
                        int64_t cap, int64_t* out_offsets, int64_t* n_ids, int64_t* bad_pos) {
  if (!E || S < 0 || !seg_off) return ORC_E_ARG;
  int64_t maxlen = 0;
  for (int64_t s = 0; s < S; s++) {
    int64_t l = seg_off[s + 1] - seg_off[s];
    if (l < 0) return ORC_E_ARG;
    if (l > maxlen) maxlen = l;
  }
  uint32_t* cps = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(maxlen + 1));
  int64_t* boff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(maxlen + 1));
  int64_t* starts = (int64_t*)malloc(sizeof(int64_t) * (size_t)(maxlen + 1));
  int64_t* chunks = (int64_t*)malloc(sizeof(int64_t) * (size_t)(maxlen + 1));
  int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)(maxlen + 1));
  if (!cps || !boff || !starts || !chunks || !scratch) {
    free(cps); free(boff); free(starts); free(chunks); free(scratch);
    return ORC_E_NOMEM;
  }
  orc_sink sink = {out, cap, 0, scratch};
  int rc = ORC_OK;
  for (int64_t s = 0; s < S && rc == ORC_OK; s++) {
    if (out_offsets) out_offsets[s] = sink.count;
    const uint8_t* seg = text + seg_off[s];
    int64_t nb = seg_off[s + 1] - seg_off[s], ncp = 0, bad = -1;
    rc = utf8_decode(seg, nb, cps, boff, &ncp, &bad);
    if (rc) {
      if (bad_pos) *bad_pos = seg_off[s] + bad;
      break;
    }
    int64_t nch = 0;
    if (tiktoken_safe && ncp > 0) {
      nch = safe_chunks(cps, ncp, chunks);
    } else {
      chunks[0] = 0;
      nch = ncp > 0 ? 1 : 0;
    }
    for (int64_t k = 0; k < nch && rc == ORC_OK; k++) {
      int64_t c0 = chunks[k], c1 = (k + 1 < nch) ? chunks[k + 1] : ncp;
      rc = encode_chunk(E, seg, cps, boff, ncp, c0, c1, allow ? allow[s] : 0, starts, &sink);
    }
  }
  if (rc == ORC_OK && out_offsets) out_offsets[S] = sink.count;
  *n_ids = sink.count;
  free(cps); free(boff); free(starts); free(chunks); free(scratch);
  if (rc == ORC_OK && sink.count > cap) rc = ORC_E_CAPACITY;
  return rc;
}

/* Pre-token boundaries of one ordinary piece of UTF-8 text, as byte offsets
 * (for tests of the split alone).  Returns the count, or a negative error. */
int64_t orc_split_bytes(const uint8_t* s, int64_t n, int64_t* byte_starts, int pattern) {
  uint32_t* cps = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(n + 1));
  int64_t* boff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int64_t* st = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!cps || !boff || !st) { free(cps); free(boff); free(st); return ORC_E_NOMEM; }
  int64_t ncp = 0, bad = -1;
  int64_t rc = utf8_decode(s, n, cps, boff, &ncp, &bad);
  if (rc == ORC_OK) {
    rc = orc_split_cps(cps, ncp, st, pattern);
    for (int64_t k = 0; k < rc; k++) byte_starts[k] = boff[st[k]];
  }
  free(cps); free(boff); free(st);
  return rc;
}

/* Byte offsets of the safe chunks of one segment (for tests). */
int64_t orc_safe_chunks_bytes(const uint8_t* s, int64_t n, int64_t* byte_starts) {
  uint32_t* cps = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)(n + 1));
  int64_t* boff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int64_t* st = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!cps || !boff || !st) { free(cps); free(boff); free(st); return ORC_E_NOMEM; }
  int64_t ncp = 0, bad = -1;
  int64_t rc = utf8_decode(s, n, cps, boff, &ncp, &bad);
  if (rc == ORC_OK) {
    rc = ncp ? safe_chunks(cps, ncp, st) : 0;
    for (int64_t k = 0; k < rc; k++) byte_starts[k] = boff[st[k]];
  }
  free(cps); free(boff); free(st);
  return rc;
}

/* ------------------------------------------------------------------------- */
/* Decode ([TT] "The byte floor": a round trip reproduces the input byte for */
/* byte; "Pitfalls that bite in production": a character's bytes may span     */
/* several ids, so the output is all ids' bytes concatenated).  Writes the    */
/* bytes of each id in turn; *len receives the total even if it exceeds cap.  */

int orc_decode(const orc_enc* E, const int32_t* ids, int64_t n, uint8_t* out, int64_t cap,
               int64_t* len) {
  int64_t k = 0;
  for (int64_t i = 0; i < n; i++) {
    const uint8_t* p = NULL;
    int64_t l = 0;
    int32_t id = ids[i];
    if (id >= 0 && id <= E->max_id && E->by_id[id] >= 0) {
      p = E->plain[E->by_id[id]].p;
      l = E->plain[E->by_id[id]].len;
    } else {
      for (int64_t s = 0; s < E->n_spec; s++)
        if (E->spec_ids[s] == id) {
          p = E->spec_bytes + E->spec_off[s];
          l = E->spec_off[s + 1] - E->spec_off[s];
        }
    }
    if (!p) { *len = k; return ORC_E_BADID; }
    for (int64_t j = 0; j < l; j++) {
      if (k < cap) out[k] = p[j];
      k++;
    }
  }
  *len = k;
  return k > cap ? ORC_E_CAPACITY : ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Streaming decode ([TT] "Pitfalls that bite in production": tokens are not   */
/* characters, so a token can end inside a character; accumulate the bytes    */
/* and hold back any trailing partial sequence).  A trailing partial sequence */
/* is a proper prefix of a well-formed UTF-8 character: a lead byte followed  */
/* by fewer continuation bytes than it announces, each in its allowed range   */
/* (Unicode's table of well-formed byte sequences: after E0 the next byte is  */
/* A0..BF, after ED 80..9F, after F0 90..BF, after F4 80..8F, else 80..BF).   */
/* Returns how many of the last bytes of b[0..n) form such a prefix (0..3).   */

static int lead_len(uint8_t b) {
  if (b >= 0xC2 && b <= 0xDF) return 2;
  if (b >= 0xE0 && b <= 0xEF) return 3;
  if (b >= 0xF0 && b <= 0xF4) return 4;
  return 0; /* ASCII, a continuation byte, or a byte that never leads */
}

static int second_ok(uint8_t lead, uint8_t b) {
  if (lead == 0xE0) return b >= 0xA0 && b <= 0xBF;
  if (lead == 0xED) return b >= 0x80 && b <= 0x9F;
  if (lead == 0xF0) return b >= 0x90 && b <= 0xBF;
  if (lead == 0xF4) return b >= 0x80 && b <= 0x8F;
  return b >= 0x80 && b <= 0xBF;
}

int orc_utf8_holdback(const uint8_t* b, int64_t n) {
  /* try each possible start of the partial character: 1, 2, 3 bytes from the end */
  for (int64_t k = 1; k <= 3 && k <= n; k++) {
    const int64_t p = n - k;
    const int need = lead_len(b[p]);
    if (need == 0) continue;  /* not a lead byte: the start must be further back */
    if (k >= need) return 0;   /* the character at p is complete (or too long) */
    for (int64_t j = p + 1; j < n; j++) {
      const int ok = (j == p + 1) ? second_ok(b[p], b[j]) : (b[j] >= 0x80 && b[j] <= 0xBF);
      if (!ok) return 0;
    }
    return (int)k;
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Plain BPE trainer for the tiny table: split the corpus with the pattern,   */
/* count identical pre-tokens, then repeatedly merge the most frequent        */
/* adjacent pair whose concatenation is not yet a token (ties: smallest       */
/* (left id, right id)); the k-th new token gets rank 256 + k.  Each round    */
/* recounts every pair from scratch.                                          */

typedef struct {
  int64_t start, len;
} orc_span;

static const uint8_t* g_corpus; /* qsort comparator context */
static int cmp_span(const void* x, const void* y) {
  const orc_span* a = (const orc_span*)x;
  const orc_span* b = (const orc_span*)y;
  return cmp_bytes(g_corpus + a->start, a->len, g_corpus + b->start, b->len);
}

/* tokens_out: bytes of tokens 256..256+n_merges-1 concatenated; tok_off[k]..
 * tok_off[k+1] delimits token 256+k (tok_off has n_merges+1 entries).
 * Returns the number of merges made (fewer if no pair is left). */
int64_t orc_train(const uint8_t* corpus, int64_t n, int64_t n_merges, uint8_t* tokens_out,
                  int64_t tokens_cap, int64_t* tok_off) {
  int64_t* bst = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!bst) return ORC_E_NOMEM;
  int64_t np = orc_split_bytes(corpus, n, bst, ORC_PATTERN_CL100K);
  if (np < 0) { free(bst); return np; }
  orc_span* sp = (orc_span*)malloc(sizeof(orc_span) * (size_t)(np ? np : 1));
  for (int64_t i = 0; i < np; i++) {
    sp[i].start = bst[i];
    sp[i].len = (i + 1 < np ? bst[i + 1] : n) - bst[i];
  }
  free(bst);
  g_corpus = corpus;
  qsort(sp, (size_t)np, sizeof(orc_span), cmp_span);
  /* unique words with counts; each word is a sequence of token ids */
  int64_t nw = 0, total_syms = 0;
  for (int64_t i = 0; i < np; i++)
    if (i == 0 || cmp_span(&sp[i - 1], &sp[i]) != 0) { nw++; total_syms += sp[i].len; }
  int64_t* wcount = (int64_t*)calloc((size_t)(nw ? nw : 1), sizeof(int64_t));
  int64_t* woff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nw + 1));
  int64_t* wlen = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nw ? nw : 1));
  int32_t* sym = (int32_t*)malloc(sizeof(int32_t) * (size_t)(total_syms ? total_syms : 1));
  int64_t w = -1, pos = 0;
  for (int64_t i = 0; i < np; i++) {
    if (i == 0 || cmp_span(&sp[i - 1], &sp[i]) != 0) {
      w++;
      woff[w] = pos;
      wlen[w] = sp[i].len;
      for (int64_t j = 0; j < sp[i].len; j++) sym[pos + j] = corpus[sp[i].start + j];
      pos += sp[i].len;
    }
    wcount[w]++;
  }
  woff[nw] = pos;
  free(sp);
  /* token bytes: ids 0..255 are the bytes, then the learned tokens */
  int64_t max_tok = 256 + n_merges;
  int64_t* tstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)max_tok);
  int64_t* tlen = (int64_t*)malloc(sizeof(int64_t) * (size_t)max_tok);
  int64_t bytes_cap = 256 + tokens_cap;
  uint8_t* tbytes = (uint8_t*)malloc((size_t)bytes_cap);
  for (int b = 0; b < 256; b++) { tbytes[b] = (uint8_t)b; tstart[b] = b; tlen[b] = 1; }
  int64_t tb_used = 256;
  /* pair counts, recounted every round in an open-addressing table whose
   * slots are cleared lazily by a round stamp; excluded pairs (their
   * concatenation already is a token) are kept in a plain list */
  const int64_t HSIZE = (int64_t)1 << 21;
  int64_t* hkey = (int64_t*)malloc(sizeof(int64_t) * (size_t)HSIZE);
  int64_t* hcnt = (int64_t*)malloc(sizeof(int64_t) * (size_t)HSIZE);
  int64_t* hstamp = (int64_t*)malloc(sizeof(int64_t) * (size_t)HSIZE);
  int64_t* touched = (int64_t*)malloc(sizeof(int64_t) * (size_t)HSIZE);
  int64_t* excl = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_merges + 1) * 64);
  int64_t n_excl = 0, excl_cap = (n_merges + 1) * 64;
  for (int64_t i = 0; i < HSIZE; i++) hstamp[i] = -1;
  int64_t made = 0;
  tok_off[0] = 0;
  for (int64_t k = 0; k < n_merges; k++) {
    int64_t ntok = 256 + made, nt = 0;
    for (int64_t wi = 0; wi < nw; wi++)
      for (int64_t j = 0; j + 1 < wlen[wi]; j++) {
        int64_t key = (int64_t)sym[woff[wi] + j] * max_tok + sym[woff[wi] + j + 1];
        uint64_t h = ((uint64_t)key * 0x9E3779B97F4A7C15ull) >> 43; /* 21 bits */
        while (hstamp[h] == k && hkey[h] != key) h = (h + 1) & (uint64_t)(HSIZE - 1);
        if (hstamp[h] != k) { hstamp[h] = k; hkey[h] = key; hcnt[h] = 0; touched[nt++] = (int64_t)h; }
        hcnt[h] += wcount[wi];
      }
    int64_t ba = -1, bb = -1, bc = 0;
    for (;;) {
      ba = -1; bc = 0;
      for (int64_t t = 0; t < nt; t++) {
        int64_t h = touched[t], key = hkey[h], c = hcnt[h];
        int64_t a = key / max_tok, b = key % max_tok;
        int skip = 0;
        for (int64_t e = 0; e < n_excl && !skip; e++) skip = (excl[e] == key);
        if (skip) continue;
        if (c > bc || (c == bc && c > 0 && (a < ba || (a == ba && b < bb)))) { bc = c; ba = a; bb = b; }
      }
      if (ba < 0) break;
      /* is the concatenation already a token? */
      int64_t cl = tlen[ba] + tlen[bb];
      int exists = 0;
      for (int64_t t = 0; t < ntok && !exists; t++)
        if (tlen[t] == cl && memcmp(tbytes + tstart[t], tbytes + tstart[ba], (size_t)tlen[ba]) == 0 &&
            memcmp(tbytes + tstart[t] + tlen[ba], tbytes + tstart[bb], (size_t)tlen[bb]) == 0)
          exists = 1;
      if (!exists) break;
      if (n_excl < excl_cap) excl[n_excl++] = ba * max_tok + bb;
    }
    if (ba < 0) break;
    int64_t cl = tlen[ba] + tlen[bb];
    if (tb_used + cl > bytes_cap) break;
    int64_t id = ntok;
    tstart[id] = tb_used;
    tlen[id] = cl;
    memcpy(tbytes + tb_used, tbytes + tstart[ba], (size_t)tlen[ba]);
    memcpy(tbytes + tb_used + tlen[ba], tbytes + tstart[bb], (size_t)tlen[bb]);
    tb_used += cl;
    memcpy(tokens_out + tok_off[made], tbytes + tstart[id], (size_t)cl);
    tok_off[made + 1] = tok_off[made] + cl;
    made++;
    /* replace the pair left to right in every word */
    for (int64_t wi = 0; wi < nw; wi++) {
      int32_t* s = sym + woff[wi];
      int64_t L = wlen[wi], o = 0;
      for (int64_t j = 0; j < L; j++) {
        if (j + 1 < L && s[j] == ba && s[j + 1] == bb) { s[o++] = (int32_t)id; j++; }
        else s[o++] = s[j];
      }
      wlen[wi] = o;
    }
  }
  free(wcount); free(woff); free(wlen); free(sym);
  free(tstart); free(tlen); free(tbytes);
  free(hkey); free(hcnt); free(hstamp); free(touched); free(excl);
  return made;
}

/* Selects the split pattern of an encoding (ORC_PATTERN_CL100K by default). */
int orc_set_pattern(orc_enc* E, int pattern) {
  if (!E || (pattern != ORC_PATTERN_CL100K && pattern != ORC_PATTERN_R50K_DIGITS)) return ORC_E_ARG;
  E->pattern = pattern;
  return ORC_OK;
}
