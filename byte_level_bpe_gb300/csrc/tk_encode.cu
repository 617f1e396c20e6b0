// tk_encode.cu -- the encode path of libtk: safe chunking, specials, split,
// byte-pair merge and ordered assembly, all as CUDA kernels (the caller's
// stream, plus two side streams for the longer pieces).
//
// Method (what is computed) follows "tiktoken Deep Dive" ("The split
// pattern", "Inside encode: a parts vector and a linear scan", "Special
// tokens ...") and "Making Kimi K3 Tokenization 18x Faster For Million Token
// Agentic Workloads" ("One native call for the whole serving path": typed
// segments, 400k / 25k safe chunking).  How it is computed is GPU-first:
//
//  * split: every byte decides on its own whether a pre-token starts there.
//    Trying the eight clauses left to right is equivalent to a start test
//    that looks at the classes of at most four preceding and one following
//    code point, plus three run-level facts: the position inside a run of
//    numbers (mod 3), whether a run of CR/LF that opens a white-space run was
//    taken by a preceding "other" run (clause 4's [\r\n]*), and whether the
//    rest of a white-space run holds a CR/LF or reaches the piece end
//    (clauses 5-7).  The number-run carry crosses tiles through a decoupled
//    look-back chain; the white-space facts are read by walking the run.
//  * merge: the parts loop over token ids (a pair of pieces merges to the
//    token whose bytes are their concatenation, looked up in a pair table
//    built at load), sized to the piece: 1-4 bytes in the tile kernel from
//    slice ranks loaded at once, 5-16 bytes one thread each over the whole
//    grid (k_merge_mid), longer pieces per warp, CTA or CTA cluster, the
//    longest in exact rounds: all leftmost-chained occurrences of the current
//    minimum-rank pair merge at once, stopping the round at the first merge
//    that creates a pair of lower rank, which is exactly the sequence the
//    one-at-a-time loop would take.  Repeated pieces of 5 bytes or more are
//    merged once per call (word caches).
//  * assembly: each 4 KiB tile stages its short ids and a table of its longer
//    pieces; after the side streams join, the table gets the pieces' counts,
//    the tile counts are scanned, and each tile's ids are written in order.
#include <stdarg.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "tk_internal.cuh"
#include "tk_unicode_table.h"

namespace tk {

// Split classes of a code point (3 bits) and flags for clause 1.
enum : uint8_t { K_L = 0, K_N = 1, K_O = 2, K_NL = 3, K_SP = 4, K_WSO = 5, K_CONT = 6, K_OUT = 7 };
enum : uint8_t { F_APOS = 0x08, F_C1 = 0x10, F_LL = 0x20, F_VR = 0x40, F_E = 0x80 };

__device__ __forceinline__ uint32_t uni_class(uint32_t cp) {
  if (cp >= 0x110000) return 0;
  const uint32_t blk = __ldg(&tk_uni_index[cp >> 8]);
  const uint32_t b = __ldg(&tk_uni_blocks[blk * 64 + ((cp & 255) >> 2)]);
  return (b >> (2 * (cp & 3))) & 3;
}

// Class and clause-1 flags of a code point.
__device__ __forceinline__ uint8_t kclass(uint32_t cp) {
  if (cp < 128) {
    if (cp == 0x20) return K_SP;
    if (cp == 0x0A || cp == 0x0D) return K_NL;
    if (cp == 0x09 || cp == 0x0B || cp == 0x0C) return K_WSO;
    const uint32_t lc = cp | 0x20;
    if (lc >= 'a' && lc <= 'z') {
      uint8_t f = 0;
      if (lc == 's' || lc == 'd' || lc == 'm' || lc == 't') f = F_C1;
      else if (lc == 'l') f = F_LL;
      else if (lc == 'v' || lc == 'r') f = F_VR;
      else if (lc == 'e') f = F_E;
      return K_L | f;
    }
    if (cp >= '0' && cp <= '9') return K_N;
    if (cp == 0x27) return K_O | F_APOS;
    return K_O;
  }
  const uint32_t u = uni_class(cp);
  if (u == 1) return cp == 0x17F ? (uint8_t)(K_L | F_C1) : (uint8_t)K_L;  // U+017F folds to s
  if (u == 2) return K_N;
  if (u == 3) return K_WSO;  // non-ASCII white space is never CR, LF or U+0020
  return K_O;
}

// Decodes the UTF-8 sequence that starts with b0; returns its length (1 when
// malformed, with ok = false).
__device__ __forceinline__ int utf8_seq(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3,
                                        uint32_t& cp, bool& ok) {
  ok = true;
  if (b0 < 0x80) { cp = b0; return 1; }
  const bool c1 = (b1 & 0xC0) == 0x80, c2 = (b2 & 0xC0) == 0x80, c3 = (b3 & 0xC0) == 0x80;
  if (b0 >= 0xC2 && b0 <= 0xDF && c1) { cp = ((b0 & 0x1F) << 6) | (b1 & 0x3F); return 2; }
  if (b0 >= 0xE0 && b0 <= 0xEF && c1 && c2) {
    cp = ((b0 & 0x0F) << 12) | ((b1 & 0x3F) << 6) | (b2 & 0x3F);
    if (cp >= 0x800 && (cp < 0xD800 || cp > 0xDFFF)) return 3;
  } else if (b0 >= 0xF0 && b0 <= 0xF4 && c1 && c2 && c3) {
    cp = ((b0 & 0x07) << 18) | ((b1 & 0x3F) << 12) | ((b2 & 0x3F) << 6) | (b3 & 0x3F);
    if (cp >= 0x10000 && cp <= 0x10FFFF) return 4;
  }
  ok = false;
  cp = 0xFFFD;
  return 1;
}

__device__ __forceinline__ bool is_ws(uint8_t k) { k &= 7; return k == K_NL || k == K_SP || k == K_WSO; }

// Python str.isspace() on a code point: \s plus U+001C..U+001F (the legacy
// chunking rule came from a Python implementation).
__device__ __forceinline__ bool py_isspace(uint32_t cp) {
  if (cp >= 0x1C && cp <= 0x1F) return true;
  if (cp < 128) return cp == 0x20 || (cp >= 0x09 && cp <= 0x0D);
  return uni_class(cp) == 3;
}

__device__ __forceinline__ bool bit_get(const uint32_t* b, int64_t i) { return (b[i >> 5] >> (i & 31)) & 1u; }

// --------------------------------------------------------------------------
// Device view of one encode call.

struct Call {
  const uint8_t* text;
  int64_t n;
  // Long pieces are indexed in the workspace by their global position
  // gb + p: a pipelined host call places batch k's text at gb inside one
  // staging buffer (text - gb), so a long piece of a later batch can use the
  // ids merged for an identical piece of an earlier one.  0 otherwise.
  int64_t gb;
  const int64_t* seg_off;
  const uint8_t* allow;
  int64_t S;
  int safe;
  Tables T;
  Work W;
};

// Index of the segment holding byte pos (largest s with seg_off[s] <= pos,
// skipping empty segments).
__device__ int64_t seg_of(const Call& c, int64_t pos) {
  int64_t lo = 0, hi = c.S - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (c.seg_off[mid] <= pos) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// First s in [0, S] with seg_off[s] >= pos.
__device__ int64_t seg_lower(const Call& c, int64_t pos) {
  int64_t lo = 0, hi = c.S + 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (c.seg_off[mid] < pos) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint8_t gbyte(const Call& c, int64_t p) {
  return (p >= 0 && p < c.n) ? __ldg(&c.text[p]) : 0;
}

// The byte at global position G (a long piece's bytes, possibly in an earlier
// batch of the same pipelined call).
__device__ __forceinline__ uint8_t text_at(const Call& c, int64_t G) { return __ldg(c.text - c.gb + G); }

__device__ bool g_chunk_cut(const Call& c, int64_t pos) {
  if (!c.safe) return false;
  return bit_get(c.W.win_cut, pos) || bit_get(c.W.run_cut, pos);
}

// Length of the longest special that starts at pos inside an allow_special
// segment, fits in the segment and crosses no chunk cut; 0 if none.  Reads
// global memory (slow path, used outside the shared-memory window).
__device__ int g_special_at(const Call& c, int64_t pos, int32_t* id) {
  if (c.T.n_spec == 0 || pos < 0 || pos >= c.n) return 0;
  const uint32_t b = gbyte(c, pos);
  if (!((c.T.spec_first[b >> 5] >> (b & 31)) & 1u)) return 0;
  const int64_t s = seg_of(c, pos);
  if (!c.allow[s]) return 0;
  const int64_t send = c.seg_off[s + 1];
  int best = 0;
  for (int k = 0; k < c.T.n_spec; k++) {
    const int L = c.T.spec_off[k + 1] - c.T.spec_off[k];
    if (L <= best || pos + L > send) continue;
    bool m = true;
    for (int j = 0; j < L && m; j++) m = gbyte(c, pos + j) == c.T.spec_bytes[c.T.spec_off[k] + j];
    for (int j = 1; j < L && m; j++) m = !g_chunk_cut(c, pos + j);
    if (m) { best = L; if (id) *id = c.T.spec_ids[k]; }
  }
  return best;
}

// Piece start at byte pos (pos is a code-point start): text start or end, a
// segment start, a chunk cut, or the start or end of a special span.
__device__ bool g_piece_start(const Call& c, int64_t pos) {
  if (pos <= 0 || pos >= c.n) return true;
  const int64_t s = seg_lower(c, pos);
  if (s <= c.S && c.seg_off[s] == pos) return true;
  if (g_chunk_cut(c, pos)) return true;
  if (c.T.n_spec == 0) return false;
  if (g_special_at(c, pos, nullptr)) return true;
  for (int k = 0; k < c.T.n_spec; k++) {
    const int L = c.T.spec_off[k + 1] - c.T.spec_off[k];
    if (pos - L >= 0 && g_special_at(c, pos - L, nullptr) == L) return true;
  }
  return false;
}

__device__ uint8_t g_kc(const Call& c, int64_t pos, int* len) {
  uint32_t cp;
  bool ok;
  const int L = utf8_seq(gbyte(c, pos), gbyte(c, pos + 1), gbyte(c, pos + 2), gbyte(c, pos + 3), cp, ok);
  if (len) *len = L;
  return kclass(cp);
}

// Start of the code point before pos (a 4-byte sequence has its lead 4 back).
__device__ int64_t g_prev(const Call& c, int64_t pos) {
  for (int k = 1; k <= 4; k++)
    if ((gbyte(c, pos - k) & 0xC0) != 0x80) return pos - k;
  return pos - 1;
}

// --------------------------------------------------------------------------
// Look-back helpers (one thread).

// Number-run carry: bit 2 = the tile is one unbroken run of numbers, bits 0-1
// = count of numbers at its end, mod 3.
struct NRunOp {
  __device__ static uint64_t id() { return 4; }
  __device__ static uint64_t reset_id() { return 0; }          // before the text: no run
  __device__ static bool resets(uint64_t v) { return !(v & 4); }
  __device__ static uint64_t comb(uint64_t l, uint64_t r) {
    if (!(r & 4)) return r;
    return (l & 4) | (((l & 3) + (r & 3)) % 3);
  }
};
// Segmented count: bit 40 = a head was seen, bits 0-39 = count since it.
struct SegCountOp {
  __device__ static uint64_t id() { return 0; }
  __device__ static uint64_t reset_id() { return 1ull << 40; }  // before the text: a head
  __device__ static bool resets(uint64_t v) { return (v >> 40) != 0; }
  __device__ static uint64_t comb(uint64_t l, uint64_t r) {
    if (r >> 40) return r;
    return (l & (1ull << 40)) | ((l & ((1ull << 40) - 1)) + r);
  }
};

// --------------------------------------------------------------------------
// Kernel: zero the status block and the look-back descriptors of one call.

__global__ void k_reset(Work W, int64_t n_desc_split, int64_t n_desc_scan, int safe,
                        int64_t n_cut_words, int64_t n_tiles, int clear_dtab) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (tid == 0) {
    Status s = {};
    s.err_pos = INT64_MAX;
    s.n_tiles = n_tiles;
    *W.status = s;
  }
  for (int64_t i = tid; i < n_tiles; i += stride) W.tile_first[i] = 0xFFFFFFFFu;  // no start yet
  for (int64_t i = tid; i < n_desc_split; i += stride) {
    W.desc_a[i] = 0;
    W.desc_b[i] = 0;
    if (safe) { W.desc_w[i] = 0; W.desc_r[i] = 0; }
  }
  for (int64_t i = tid; i < n_desc_scan; i += stride) W.desc_c[i] = 0;
  if (safe)
    for (int64_t i = tid; i < n_cut_words; i += stride) { W.win_cut[i] = 0; W.run_cut[i] = 0; }
  if (clear_dtab)
    for (int64_t i = tid; i < (2ll << W.dtab_log2); i += stride) W.dtab[i] = 0ull;
}

// Segment table check: seg_off[0] = 0, non-decreasing, seg_off[S] = n.
__global__ void k_check_segments(Call c) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (int64_t s = tid; s <= c.S; s += (int64_t)gridDim.x * blockDim.x) {
    const int64_t v = c.seg_off[s];
    bool bad = (s == 0 && v != 0) || (s == c.S && v != c.n) || v < 0 || v > c.n;
    if (s > 0 && c.seg_off[s - 1] > v) bad = true;
    if (bad) set_error(c.W.status, TK_E_ARG, 1);
  }
}

// Per split tile, the first segment index at or after t0 - HALO, t0,
// t0 + TILE and t0 + TILE + HALO (four binary searches per tile, in parallel,
// so that no tile kernel searches on its critical path).
__global__ void k_tile_segs(Call c) {
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < 4 * ntiles;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i >> 2, k = i & 3;
    const int64_t pos = tile * TILE + (k == 0 ? -HALO : k == 1 ? 0 : k == 2 ? TILE : TILE + HALO);
    c.W.tile_segs[i] = (uint32_t)seg_lower(c, pos);
  }
}

// --------------------------------------------------------------------------
// Safe chunking: a segmented count of code points over the text.
//   mode 0 (windows): heads are segment starts; a cut goes before every code
//     point whose index since the head is a positive multiple of 400,000.
//   mode 1 (runs): heads are segment starts, window cuts and changes of
//     isspace(); a cut goes before every code point whose index in its run is
//     a positive multiple of 25,000.
// Tiles of 4 KiB, 256 threads x 16 bytes, persistent with dynamic tiles.

__global__ void __launch_bounds__(SPLIT_THREADS) k_chunk_scan(Call c, int mode) {
  constexpr int CB = 16;  // bytes loaded before the tile (a 16-byte aligned window)
  __shared__ __align__(16) uint8_t s_text[TILE + 2 * CB];
  __shared__ uint32_t s_head[TILE / 32];  // segment starts (and window cuts in mode 1)
  __shared__ uint64_t s_wtot[SPLIT_THREADS / 32];
  __shared__ int64_t s_tile;
  __shared__ uint64_t s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const bool aligned = ((uintptr_t)c.text & 15) == 0;
  uint64_t* desc = mode == 0 ? c.W.desc_w : c.W.desc_r;
  uint32_t* out = mode == 0 ? c.W.win_cut : c.W.run_cut;
  const int64_t M = mode == 0 ? CHUNK_CHARS : RUN_CHARS;
  for (;;) {
    if (tid == 0) s_tile = atomicAdd(&c.W.status->tile_ctr[1 + mode], 1u);
    __syncthreads();
    const int64_t tile = s_tile;
    if (tile >= ntiles) break;
    const int64_t t0 = tile * TILE;
    // bytes [t0 - CB, t0 + TILE + CB), 16 at a time where they lie in the text
    for (int v = tid; v < (TILE + 2 * CB) / 16; v += SPLIT_THREADS) {
      const int64_t p = t0 - CB + 16 * v;
      if (aligned && p >= 0 && p + 16 <= c.n) {
        *reinterpret_cast<uint4*>(&s_text[16 * v]) = ld_na_v4(c.text + p);
      } else {
        for (int j = 0; j < 16; j++) s_text[16 * v + j] = gbyte(c, p + j);
      }
    }
    // heads known before the scan: segment starts (the text start among
    // them), and in mode 1 the window cuts
    for (int i = tid; i < TILE / 32; i += SPLIT_THREADS) {
      uint32_t v = 0;
      if (mode == 1 && t0 + 32 * i < c.n) v = c.W.win_cut[(t0 >> 5) + i];
      s_head[i] = v;
    }
    __syncthreads();
    {
      const int64_t slo = c.W.tile_segs[4 * tile + 1], shi = c.W.tile_segs[4 * tile + 2];
      for (int64_t sg = slo + tid; sg < shi; sg += SPLIT_THREADS) {
        const int64_t x = c.seg_off[sg] - t0;
        if (x >= 0 && x < TILE) atomicOr(&s_head[x >> 5], 1u << (x & 31));
      }
      if (tid == 0 && t0 == 0) atomicOr(&s_head[0], 1u);
    }
    __syncthreads();
    // per-thread aggregate over its 16 bytes
    const int xb = CB + tid * 16;
    uint64_t agg = 0;
    uint32_t heads = (s_head[tid >> 1] >> (16 * (tid & 1))) & 0xFFFFu;
    uint32_t starts = 0;  // bit j: byte xb + j is a head / code-point start
    for (int j = 0; j < 16; j++) {
      const int x = xb + j;
      const int64_t pos = t0 + tid * 16 + j;
      if (pos >= c.n) break;
      const uint32_t b = s_text[x];
      if ((b & 0xC0) == 0x80) continue;
      starts |= 1u << j;
      bool head = (heads >> j) & 1u;
      if (mode == 1 && !head) {
        uint32_t cp, pcp;
        bool ok;
        utf8_seq(b, s_text[x + 1], s_text[x + 2], s_text[x + 3], cp, ok);
        int px = x - 1;
        while (px > x - 4 && (s_text[px] & 0xC0) == 0x80) px--;
        utf8_seq(s_text[px], s_text[px + 1], s_text[px + 2], s_text[px + 3], pcp, ok);
        head = py_isspace(cp) != py_isspace(pcp);
        if (head) heads |= 1u << j;
      }
      if (head) agg = 1ull << 40;
      agg += 1;
    }
    heads &= starts;
    // exclusive scan of the thread aggregates: warp shuffles, then the warps
    uint64_t inc = agg;
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc = SegCountOp::comb(y, inc);
    }
    if (lane == 31) s_wtot[warp] = inc;
    __syncthreads();
    if (tid < 32) {
      uint64_t run = SegCountOp::id();
      for (int w = 0; w < SPLIT_THREADS / 32; w++) run = SegCountOp::comb(run, s_wtot[w]);
      if (tid == 0) st_release_u64(&desc[tile], DESC_AGG | run);
      const uint64_t carry = carry_walk_warp<SegCountOp>(desc, tile, run, c.W.status, 2 + mode);
      if (tid == 0) s_carry = carry;
    }
    __syncthreads();
    uint64_t pre = s_carry;
    for (int w = 0; w < warp; w++) pre = SegCountOp::comb(pre, s_wtot[w]);
    uint64_t e = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) e = SegCountOp::id();
    const uint64_t v = SegCountOp::comb(pre, e);
    int64_t idx = (int64_t)(v & ((1ull << 40) - 1));
    for (uint32_t bits = starts; bits; bits &= bits - 1) {
      const int j = __ffs(bits) - 1;
      if ((heads >> j) & 1u) idx = 0;
      if (idx > 0 && idx % M == 0) {
        const int64_t pos = t0 + tid * 16 + j;
        atomicOr(&out[pos >> 5], 1u << (pos & 31));
      }
      idx++;
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------------------
// Split kernel: per 4 KiB tile, pre-token starts -> ordered records.

constexpr int WSEG_MAX = 64;
constexpr int WALK_MAX = 32;
constexpr uint32_t NRUN_WALK = 32;  // numbers a thread walks back over before the block scan
struct SplitSmem {
  uint8_t text[WIN + 16];
  uint8_t kc[WIN];
  uint32_t pst[WIN / 32];   // piece starts
  uint32_t insp[WIN / 32];  // bytes inside special spans
  uint32_t sst[WIN / 32];   // special span starts
  // the segments that meet the window (at most WSEG_MAX): their starts
  // relative to the window (-1: before it), one more entry for the end of the
  // last, and their allow_special flags; nwseg = -1 when there are more
  int32_t wseg[WSEG_MAX + 1];
  uint8_t wallow[WSEG_MAX];
  int nwseg;
  uint32_t scan[SPLIT_THREADS / 32];  // number runs: the warps' aggregates (long runs only)
  // white-space walks past the window, deferred to a warp each (walk_rest)
  int nreq;
  int64_t req_q[WALK_MAX];
  uint16_t req_owner[WALK_MAX];  // thread << 4 | bit
  uint8_t req_check[WALK_MAX];
  uint8_t req_res[WALK_MAX];
  int64_t tile;
  int64_t seg[2];
  uint64_t ncarry;
};
static_assert(offsetof(SplitSmem, kc) % 4 == 0, "class bytes are read as words");

// Special match of the longest special at window position x (all bytes must be
// in the window); returns its length or 0.
__device__ int win_special(const Call& c, const SplitSmem& sm, int x, int64_t pos) {
  const uint32_t b = sm.text[x];
  if (!((c.T.spec_first[b >> 5] >> (b & 31)) & 1u)) return 0;
  int64_t send;
  if (sm.nwseg > 0) {
    // the window's own segment table (shared memory)
    int e = sm.nwseg - 1;
    while (e > 0 && sm.wseg[e] > x) e--;
    if (!sm.wallow[e]) return 0;
    send = pos - x + sm.wseg[e + 1];
  } else {
    const int64_t s = seg_of(c, pos);
    if (!c.allow[s]) return 0;
    send = c.seg_off[s + 1];
  }
  int best = 0;
  for (int k = 0; k < c.T.n_spec; k++) {
    const int L = c.T.spec_off[k + 1] - c.T.spec_off[k];
    if (L <= best || pos + L > send || x + L > WIN) continue;
    bool m = true;
    for (int j = 0; j < L && m; j++) m = sm.text[x + j] == c.T.spec_bytes[c.T.spec_off[k] + j];
    // chunk cuts strictly inside the span forbid the match (pst holds only
    // segment starts and chunk cuts at this point)
    for (int j = 1; j < L && m; j++) m = !bit_get(sm.pst, x + j);
    if (m) best = L;
  }
  return best;
}

// The rest of a white-space run from byte q, past the shared-memory window:
// true iff the run holds no CR/LF and ends at a code point that is not white
// space inside the same piece (the clause 5-7 question).  A byte scan: the
// segment's end is looked up once; every position is first tested for a piece
// start (a chunk cut, or a special that starts there), then classified.
// check_q: whether q itself must be tested for a piece start.
__device__ bool g_ws_rest_ends_in_piece(const Call& c, int64_t q, bool check_q) {
  const int64_t seg_end = c.seg_off[seg_of(c, q) + 1];
  const int64_t lim = min(c.n, seg_end);
  // 16 bytes at a time through runs of ASCII space / tab / VT / FF: none can be
  // a CR/LF or end the run; only a chunk cut or a special can end the piece
  // there (specials are ruled out when none starts with those bytes)
  const bool ws_specials = c.T.n_spec && (((c.T.spec_first[0x20 >> 5] >> (0x20 & 31)) |
                                            (c.T.spec_first[0] >> 0x09) | (c.T.spec_first[0] >> 0x0B) |
                                            (c.T.spec_first[0] >> 0x0C)) & 1u);
  const bool vec = !ws_specials && (((uintptr_t)c.text & 15) == 0);
  for (bool first = true;; first = false) {
    if (q >= lim) return false;
    if (vec && !first && (q & 15) == 0 && q + 16 <= lim) {
      const uint4 v = *reinterpret_cast<const uint4*>(c.text + q);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      bool all_ws = true;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint32_t e = __vcmpeq4(wv[k], 0x20202020u) | __vcmpeq4(wv[k], 0x09090909u) |
                           __vcmpeq4(wv[k], 0x0B0B0B0Bu) | __vcmpeq4(wv[k], 0x0C0C0C0Cu);
        all_ws &= e == 0xFFFFFFFFu;
      }
      uint32_t cuts = 0;
      if (c.safe) cuts = ((c.W.win_cut[q >> 5] | c.W.run_cut[q >> 5]) >> (q & 31)) & 0xFFFFu;
      if (all_ws && cuts == 0) {
        q += 16;
        continue;
      }
    }
    if (!first || check_q) {
      if (g_chunk_cut(c, q)) return false;
      if (c.T.n_spec && g_special_at(c, q, nullptr)) return false;
    }
    const uint32_t b = gbyte(c, q);
    if (b == 0x0A || b == 0x0D) return false;
    if (b == 0x20 || b == 0x09 || b == 0x0B || b == 0x0C) { q++; continue; }
    if (b < 0x80) return true;
    int len;
    const uint8_t k = g_kc(c, q, &len) & 7;
    if (k != K_SP && k != K_WSO && k != K_NL) return true;
    q += len;
  }
}

// g_ws_rest_ends_in_piece run by one warp (all 32 lanes, same arguments): the
// bytes up to the next 16-byte boundary one by one (lane 0), then 512 bytes
// per step, each lane testing 16 bytes for plain white space (space, tab,
// VT, FF) with no chunk cut; from the first chunk that is not plain, lane 0
// walks on one by one.  Only when no special starts with those bytes and the
// text is 16-byte aligned, else lane 0 walks the whole way.
__device__ bool warp_ws_rest(const Call& c, int64_t q, bool check_q) {
  const int lane = threadIdx.x & 31;
  const bool ws_specials = c.T.n_spec && (((c.T.spec_first[0x20 >> 5] >> (0x20 & 31)) |
                                            (c.T.spec_first[0] >> 0x09) | (c.T.spec_first[0] >> 0x0B) |
                                            (c.T.spec_first[0] >> 0x0C)) & 1u);
  const bool vec = !ws_specials && (((uintptr_t)c.text & 15) == 0);
  int res = -1;  // lane 0: the answer once known
  int64_t a0 = (q + 16) & ~(int64_t)15;
  int64_t lim = 0;
  if (lane == 0) {
    lim = min(c.n, c.seg_off[seg_of(c, q) + 1]);
    if (!vec || a0 + 16 > lim) {
      res = g_ws_rest_ends_in_piece(c, q, check_q) ? 1 : 0;
    } else {
      // the bytes before a0, one by one: an answer there ends the walk
      int64_t p = q;
      for (bool first = true; p < a0; first = false) {
        if (!first || check_q) {
          if (g_chunk_cut(c, p)) { res = 0; break; }
          if (c.T.n_spec && g_special_at(c, p, nullptr)) { res = 0; break; }
        }
        const uint32_t b = gbyte(c, p);
        if (b == 0x0A || b == 0x0D) { res = 0; break; }
        if (b == 0x20 || b == 0x09 || b == 0x0B || b == 0x0C) { p++; continue; }
        if (b < 0x80) { res = 1; break; }
        // a multi-byte code point: the serial walk from here
        res = g_ws_rest_ends_in_piece(c, p, !first || check_q) ? 1 : 0;
        break;
      }
    }
  }
  res = __shfl_sync(0xffffffffu, res, 0);
  if (res >= 0) return res != 0;
  lim = __shfl_sync(0xffffffffu, lim, 0);
  int64_t b = lim;
  for (int64_t p = a0; p < lim; p += 512) {
    const int64_t mine = p + 16 * lane;
    bool plain = false;
    if (mine + 16 <= lim) {
      const uint4 v = *reinterpret_cast<const uint4*>(c.text + mine);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      plain = true;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint32_t e = __vcmpeq4(wv[k], 0x20202020u) | __vcmpeq4(wv[k], 0x09090909u) |
                           __vcmpeq4(wv[k], 0x0B0B0B0Bu) | __vcmpeq4(wv[k], 0x0C0C0C0Cu);
        plain &= e == 0xFFFFFFFFu;
      }
      if (plain && c.safe)
        plain = (((c.W.win_cut[mine >> 5] | c.W.run_cut[mine >> 5]) >> (mine & 31)) & 0xFFFFu) == 0;
    }
    const uint32_t np = __ballot_sync(0xffffffffu, !plain);
    if (np) {
      b = p + 16 * (__ffs(np) - 1);
      break;
    }
  }
  // [a0, b) is plain white space inside the piece: walk on from b
  if (lane == 0) res = (b < lim && g_ws_rest_ends_in_piece(c, b, true)) ? 1 : 0;
  return __shfl_sync(0xffffffffu, res, 0) != 0;
}

// Accessors that read the window when the position is trusted, else global.
struct Win {
  const Call& c;
  SplitSmem& sm;
  int64_t wlo;
  int owner;  // thread << 4 | bit of the code point under test (for deferred walks)
  int* ndef;  // this thread's count of deferred walks
  // The rest of a white-space run past the window (g_ws_rest_ends_in_piece):
  // queued for a warp (provisional answer false, fixed after the queue runs),
  // or walked here when the queue is full.
  __device__ bool walk(int64_t q, bool check_q) const {
    const int k = atomicAdd(&sm.nreq, 1);
    if (k < WALK_MAX) {
      (*ndef)++;
      sm.req_q[k] = q;
      sm.req_owner[k] = (uint16_t)owner;
      sm.req_check[k] = check_q ? 1 : 0;
      return false;
    }
    return g_ws_rest_ends_in_piece(c, q, check_q);
  }
  __device__ bool trusted(int64_t p) const {
    return p >= wlo + TRUST && p < wlo + WIN - TRUST;
  }
  __device__ uint8_t kc(int64_t p) const {
    if (trusted(p)) return sm.kc[p - wlo];
    if (p < 0 || p >= c.n) return K_OUT;
    return g_kc(c, p, nullptr);
  }
  __device__ bool pst(int64_t p) const {
    if (trusted(p)) return bit_get(sm.pst, p - wlo);
    return g_piece_start(c, p);
  }
  __device__ int64_t prev(int64_t p) const {
    if (trusted(p) && trusted(p - 4)) {
      for (int k = 1; k <= 4; k++)
        if ((sm.kc[p - k - wlo] & 7) != K_CONT) return p - k;
      return p - 1;
    }
    return g_prev(c, p);
  }
  // From q (a trusted position whose window index is a multiple of 4), past
  // every 16-byte block that holds only ASCII space, tab, VT or FF (class
  // bytes K_SP / K_WSO, no flags) with no piece start at the 16 positions
  // after q's first byte; returns the first position not skipped.
  __device__ int64_t skip_plain_ws(int64_t q) const {
    for (;;) {
      const int i = (int)(q - wlo);
      if ((i & 3) || !trusted(q) || !trusted(q + 20)) return q;
      const uint32_t* kw = reinterpret_cast<const uint32_t*>(&sm.kc[i]);
      const bool ws = ((kw[0] & 0xFEFEFEFEu) == 0x04040404u) & ((kw[1] & 0xFEFEFEFEu) == 0x04040404u) &
                      ((kw[2] & 0xFEFEFEFEu) == 0x04040404u) & ((kw[3] & 0xFEFEFEFEu) == 0x04040404u);
      if (!ws) return q;
      const int j = i + 1;  // piece starts at i + 1 .. i + 16
      const uint64_t pw = ((uint64_t)sm.pst[(j >> 5) + 1] << 32) | sm.pst[j >> 5];
      if ((pw >> (j & 31)) & 0xFFFFu) return q;
      q += 16;
    }
  }
  __device__ int64_t next(int64_t p) const {
    if (trusted(p) && trusted(p + 4)) {
      for (int k = 1; k <= 4; k++)
        if ((sm.kc[p + k - wlo] & 7) != K_CONT) return p + k;
      return p + 1;
    }
    int L;
    g_kc(c, p, &L);
    return p + L;
  }
};

// Clause 1 at an apostrophe at j: the apostrophe starts a pre-token unless it
// continues an "other" run or follows a space that starts one.
__device__ __forceinline__ bool apos_starts(const Win& w, int64_t j) {
  if (w.pst(j)) return true;
  const uint8_t p = w.kc(w.prev(j)) & 7;
  return p != K_O && p != K_SP;
}

// The start test.  x is a code-point start of ordinary text that is not a
// piece start; nidx is its index inside its run of numbers (mod 3).
__device__ bool starts_here(const Win& w, int64_t x, uint8_t kx, uint32_t nidx) {
  const int64_t p1 = w.prev(x);
  const uint8_t kp = w.kc(p1);
  const uint8_t P = kp & 7, C = kx & 7;
  switch (C) {
    case K_N:
      // r50k's digit clause " ?\p{N}++": one run, a single space before it joins
      if (w.c.T.pattern == TK_PATTERN_R50K_DIGITS) return P != K_N && P != K_SP;
      return P != K_N || nidx == 0;
    case K_L: {
      if (P == K_N || P == K_NL) return true;
      if (P == K_SP || P == K_WSO) return false;
      if (P == K_O) {
        if (w.pst(p1)) return false;
        const uint8_t P2 = w.kc(w.prev(p1)) & 7;
        return P2 == K_O || P2 == K_SP;
      }
      // P == K_L: a start only right after a clause-1 contraction
      if (w.pst(p1)) return false;
      const int64_t p2 = w.prev(p1);
      const uint8_t k2 = w.kc(p2);
      if ((k2 & F_APOS) && (kp & F_C1) && apos_starts(w, p2)) return true;
      if (w.pst(p2)) return false;
      const int64_t p3 = w.prev(p2);
      const uint8_t k3 = w.kc(p3);
      if ((k3 & F_APOS) && (((k2 & F_LL) && (kp & F_LL)) || ((k2 & F_VR) && (kp & F_E))) &&
          (k2 & 7) == K_L && apos_starts(w, p3))
        return true;
      return false;
    }
    case K_O:
      return P == K_L || P == K_N || P == K_NL || P == K_WSO;
    case K_NL:
      return P == K_L || P == K_N;
    default: {  // K_SP, K_WSO
      if (P == K_L || P == K_N || P == K_O) return true;
      if (P == K_NL) {
        // taken by a preceding other-run's [\r\n]*?  walk back over CR/LF
        int64_t j = p1;
        bool absorbed;
        for (;;) {
          if ((w.kc(j) & 7) != K_NL) { absorbed = (w.kc(j) & 7) == K_O; break; }
          if (w.pst(j)) { absorbed = false; break; }
          j = w.prev(j);
        }
        if (absorbed) return true;
        // else a start iff the rest of the run has no CR/LF and does not reach the piece end
        int64_t q = x;
        bool check_q = false;
        for (;;) {
          q = w.skip_plain_ws(q);
          if (!w.trusted(q) || !w.trusted(q + 4)) return w.walk(q, check_q);
          const uint8_t kq = w.kc(q) & 7;
          if (kq == K_NL) return false;
          if (kq != K_SP && kq != K_WSO) return true;
          q = w.next(q);
          if (q >= w.c.n) return false;
          if (!w.trusted(q)) { check_q = true; continue; }
          if (w.pst(q)) return false;
        }
      }
      // P is white space but not CR/LF: a start iff the next code point is in
      // the piece and is not white space
      const int64_t n1 = w.next(x);
      if (n1 >= w.c.n || w.pst(n1)) return false;
      return !is_ws(w.kc(n1));
    }
  }
}

// The 8x8 bit matrix of eight bytes (byte k = row k) transposed by three
// delta swaps: afterwards byte i holds bit i of every byte (bit k from byte
// k), i.e. the eight bit-planes of the eight bytes at once.
__device__ __forceinline__ uint64_t transpose8x8(uint64_t x) {
  uint64_t t;
  t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
  x = x ^ t ^ (t << 7);
  t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
  x = x ^ t ^ (t << 14);
  t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
  x = x ^ t ^ (t << 28);
  return x;
}

// The start test for 16 ASCII code points at once (window bytes x0 .. x0+15,
// no special span byte within 4 before and 4 after).  Bit k of each mask is
// window byte x0 - 4 + k; PS holds the piece starts (segment starts, chunk
// cuts) of those 24 bytes.  The rules are those of starts_here, with the number
// groups found by propagating run starts in steps of 3, and a piece start as a
// barrier: it is a start itself, no look-back reaches past it (a run of
// numbers restarts there, the other-prefix and contraction rules stop at it)
// and white space whose next code point starts another piece reaches its
// piece's end.  r is the index in its number run of the code point at x0.
// Returns the start bits of the 16 bytes; *slow receives the bytes whose test
// needs the white-space walks (CR/LF followed by other white space).
__device__ __forceinline__ uint32_t starts_ascii16(const uint32_t P[8], uint32_t r, uint32_t PS, uint32_t* slow,
                                                   bool r50k_digits) {
  const uint32_t p0 = P[0], p1 = P[1], p2 = P[2];
  const uint32_t L = ~p0 & ~p1 & ~p2, N = p0 & ~p1 & ~p2, O = ~p0 & p1 & ~p2, NL = p0 & p1 & ~p2;
  const uint32_t SP = ~p0 & ~p1 & p2, WSO = p0 & ~p1 & p2;
  const uint32_t APOS = P[3], C1 = P[4], LLf = P[5], VR = P[6], E = P[7];
  const uint32_t SPW = SP | WSO, WS = NL | SPW, OS = O | SP;
  uint32_t S_N;
  if (r50k_digits) {
    // one start per digit run, on the space before it if there is one
    S_N = N & ~(N << 1) & ~(SP << 1);
  } else {
    // numbers: group starts at run start + 3k; a number that starts a piece
    // starts a run, and only numbers that are no piece start continue one
    const uint32_t NR = N & ~PS;
    uint32_t G = (N & ~(N << 1) & ~1u) | (N & PS);
    if ((N >> 4) & (N >> 3) & ~(PS >> 4) & 1u) {  // the run at x0 began earlier: its index there is r
      const int first = 4 + (int)((3u - r) % 3u);
      const uint32_t span = ((2u << first) - 1u) & ~0xFu;  // bits 4..first
      if ((NR & span) == span) G |= 1u << first;
    }
#pragma unroll
    for (int it = 0; it < 7; it++) G |= (G << 3) & NR & (NR << 1) & (NR << 2);
    S_N = G & N;
  }
  const uint32_t nps1 = ~(PS << 1);
  const uint32_t S_L =
      L & ((N << 1) | (NL << 1) | ((O << 1) & (OS << 2) & nps1) |
           ((L << 1) & (C1 << 1) & (APOS << 2) & nps1 & (~(OS << 3) | (PS << 2))) |
           ((L << 1) & (APOS << 3) & (((LLf << 2) & (LLf << 1)) | ((VR << 2) & (E << 1))) & nps1 & ~(PS << 2) &
            (~(OS << 4) | (PS << 3))));
  const uint32_t S_O = O & ((L | N | NL | WSO) << 1);
  const uint32_t S_NL = NL & ((L | N) << 1);
  const uint32_t S_W = SPW & (((L | N | O) << 1) | ((SPW << 1) & ~(WS >> 1) & ~(PS >> 1)));
  // white space right after CR/LF: a start iff the CR/LF run before it (no
  // piece start in it) follows an "other" byte (clause 4 took it), else iff
  // the first byte after it that is not space / other white space, or is a
  // piece start, is neither a piece start nor CR/LF (the run ends inside the
  // piece without another CR/LF).  Decided here when both facts lie inside
  // the 24 bytes (segmented propagations by doubling); the rest is left to
  // starts_here.
  const uint32_t sl = SPW & (NL << 1) & ~PS;
  uint32_t nl_start = 0, nl_known = 0;
  if (sl & 0xFFFF0u) {
    const uint32_t M = NL & ~PS;
    uint32_t R = M & (O << 1), U = M & 1u, Mk = M;  // runs after "other"; runs reaching bit 0
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      R |= (R << d) & Mk;
      U |= (U << d) & Mk;
      Mk &= Mk << d;
    }
    const uint32_t absorbed = R << 1, unknown = U << 1;
    const uint32_t Z = (~SPW | PS) & 0xFFFFFFu;   // stops
    const uint32_t V = Z & ~WS & ~PS;             // stops that make a start
    uint32_t Y = (V >> 1) & (Z >> 1), K = Z >> 1;  // the first stop after each byte: known, value
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      Y |= ~K & (Y >> d);
      K |= K >> d;
    }
    nl_known = sl & ~unknown & (absorbed | K);
    nl_start = nl_known & (absorbed | Y);
  }
  *slow = ((sl & ~nl_known) >> 4) & 0xFFFFu;
  return ((((S_N | S_L | S_O | S_NL | S_W) & ~sl) | PS | nl_start) >> 4) & 0xFFFFu;
}

__global__ void __launch_bounds__(SPLIT_THREADS, 6) k_split(Call c) {
  __shared__ SplitSmem sm;
  __shared__ uint8_t s_asc[128];
  __shared__ int s_any_allow;
  const int tid = threadIdx.x;
  if (tid < 128) s_asc[tid] = kclass((uint32_t)tid);
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const bool aligned = ((uintptr_t)c.text & 15) == 0;
  for (;;) {
    if (tid == 0) {
      sm.tile = atomicAdd(&c.W.status->tile_ctr[0], 1u);
      s_any_allow = 0;
      sm.nreq = 0;
    }
    __syncthreads();
    const int64_t tile = sm.tile;
    if (tile >= ntiles) break;
    const int64_t t0 = tile * TILE;
    const int64_t wlo = t0 - HALO;
    // 1. window bytes
    for (int v = tid; v < (WIN + 16) / 16; v += SPLIT_THREADS) {
      const int64_t p = wlo + 16 * v;
      if (aligned && p >= 0 && p + 16 <= c.n) {
        *reinterpret_cast<uint4*>(&sm.text[16 * v]) = ld_na_v4(c.text + p);
      } else {
        for (int j = 0; j < 16; j++) sm.text[16 * v + j] = gbyte(c, p + j);
      }
    }
    for (int i = tid; i < WIN / 32; i += SPLIT_THREADS) {
      sm.insp[i] = 0;
      sm.sst[i] = 0;
      uint32_t v = 0;
      const int64_t word = (wlo >> 5) + i;
      if (c.safe && word >= 0 && (word << 5) < c.n) v = c.W.win_cut[word] | c.W.run_cut[word];
      sm.pst[i] = v;
    }
    const int64_t seg_lo = c.W.tile_segs[4 * tile], seg_hi = c.W.tile_segs[4 * tile + 3];
    __syncthreads();
    // 2. segment starts (and the text end) are piece starts; note whether any
    //    segment overlapping the window allows specials
    for (int64_t s = seg_lo + tid; s < seg_hi; s += SPLIT_THREADS) {
      const int64_t x = c.seg_off[s] - wlo;
      if (x >= 0 && x < WIN) atomicOr(&sm.pst[x >> 5], 1u << (x & 31));
      if (s < c.S && c.allow[s]) s_any_allow = 1;
    }
    if (tid == 0 && seg_lo > 0 && c.allow[seg_lo - 1]) s_any_allow = 1;
    {
      // segments from the one holding the window's first byte to the last that starts in it
      const int64_t sb = seg_lo > 0 ? seg_lo - 1 : 0;
      const int64_t ne = seg_hi - sb;
      const bool fits = ne >= 1 && ne <= WSEG_MAX;
      if (tid == 0) sm.nwseg = fits ? (int)ne : -1;
      if (fits)
        for (int64_t e = tid; e <= ne; e += SPLIT_THREADS) {
          const int64_t s = sb + e;
          const int64_t rel = c.seg_off[s < c.S ? s : c.S] - wlo;
          sm.wseg[e] = (int32_t)(rel < -1 ? -1 : rel);
          if (e < ne) sm.wallow[e] = (s < c.S) ? c.allow[s] : 0;
        }
    }
    __syncthreads();
    // 3. specials in allow_special segments: find, then mark
    if (c.T.n_spec > 0 && s_any_allow) {
      for (int x = tid; x < WIN; x += SPLIT_THREADS) {
        const int64_t pos = wlo + x;
        if (pos < 0 || pos >= c.n) continue;
        if (win_special(c, sm, x, pos)) atomicOr(&sm.sst[x >> 5], 1u << (x & 31));
      }
      __syncthreads();
      for (int x = tid; x < WIN; x += SPLIT_THREADS) {
        if (!bit_get(sm.sst, x)) continue;
        const int L = win_special(c, sm, x, wlo + x);
        atomicOr(&sm.pst[x >> 5], 1u << (x & 31));
        if (x + L < WIN) atomicOr(&sm.pst[(x + L) >> 5], 1u << ((x + L) & 31));
        for (int j = 0; j < L; j++) atomicOr(&sm.insp[(x + j) >> 5], 1u << ((x + j) & 31));
      }
    }
    // 4. classes (and UTF-8 validation of the tile's own bytes): four bytes at
    //    a time where all four are ASCII text, else one by one
    for (int x4 = tid; 4 * x4 < WIN; x4 += SPLIT_THREADS) {
      const int64_t pos4 = wlo + 4 * x4;
      const uint32_t tw = reinterpret_cast<const uint32_t*>(sm.text)[x4];
      if (pos4 >= 0 && pos4 + 4 <= c.n && (tw & 0x80808080u) == 0) {
        reinterpret_cast<uint32_t*>(sm.kc)[x4] =
            (uint32_t)s_asc[tw & 0x7F] | ((uint32_t)s_asc[(tw >> 8) & 0x7F] << 8) |
            ((uint32_t)s_asc[(tw >> 16) & 0x7F] << 16) | ((uint32_t)s_asc[tw >> 24] << 24);
        continue;
      }
      for (int x = 4 * x4; x < 4 * x4 + 4; x++) {
      const int64_t pos = wlo + x;
      const uint32_t b = sm.text[x];
      uint8_t k;
      if (pos < 0 || pos >= c.n) {
        k = K_OUT;
      } else if (b < 0x80) {
        k = s_asc[b];
      } else if ((b & 0xC0) == 0x80) {
        k = K_CONT;
        if (x >= HALO && x < HALO + TILE) {
          // a continuation byte must be covered by a valid sequence
          int j = x - 1;
          while (j > x - 4 && (sm.text[j] & 0xC0) == 0x80) j--;
          uint32_t cp;
          bool ok;
          const int L = utf8_seq(sm.text[j], sm.text[j + 1], sm.text[j + 2], sm.text[j + 3], cp, ok);
          if ((sm.text[j] & 0xC0) == 0x80 || !ok || j + L <= x || wlo + j < 0) {
            set_error(c.W.status, TK_E_UTF8, 0);
            atomicMin((long long*)&c.W.status->err_pos, (long long)pos);
          }
        }
      } else {
        uint32_t cp;
        bool ok;
        utf8_seq(b, sm.text[x + 1], sm.text[x + 2], sm.text[x + 3], cp, ok);
        if (!ok && x >= HALO && x < HALO + TILE) {
          set_error(c.W.status, TK_E_UTF8, 0);
          atomicMin((long long*)&c.W.status->err_pos, (long long)pos);
        }
        k = kclass(cp);
      }
      sm.kc[x] = k;
      }
    }
    __syncthreads();
    // 5. number runs.  The start test needs, for this thread's first code
    //    point, how many numbers of the same run precede it (mod 3): a walk
    //    back over the numbers before it (runs are short), stopping at a reset
    //    (a code point that is not a number, a number inside a special, or a
    //    number that starts a piece) or at the tile start.  A walk that reaches
    //    the tile start adds the tile's carry: the run that ends before t0,
    //    counted in the window if it starts there, else taken from the
    //    look-back chain over the tiles' aggregates.  Every tile publishes its
    //    aggregate (NRunOp: the numbers at its end since its last reset, and
    //    whether nothing in it resets) before anything waits on the chain.
    const int xb = HALO + tid * 16;
    int unres = 0;  // a walk gave up (a long run of numbers): block scan below
    if (tid == SPLIT_THREADS - 1) {
      int p = HALO + (int)min((int64_t)TILE, c.n - t0) - 1;
      while (p >= HALO && (sm.kc[p] & 7) == K_CONT) p--;
      uint32_t cnt = 0, unbroken = 1;
      while (p >= HALO) {
        if ((sm.kc[p] & 7) != K_N || bit_get(sm.insp, p)) { unbroken = 0; break; }
        cnt++;
        if (bit_get(sm.pst, p)) { unbroken = 0; break; }
        if (cnt == NRUN_WALK) { unres = 1; break; }  // published after the block scan
        const int q = p;
        p--;
        while (p > q - 4 && (sm.kc[p] & 7) == K_CONT) p--;
      }
      if (!unres) st_relaxed_u64(&c.W.desc_a[tile], DESC_AGG | (unbroken ? 4u : 0u) | (cnt % 3u));
    }
    const int agg_late = unres;
    uint32_t r = 0;
    int reach_t0 = 0;  // the walk ran past the tile start without a reset
    {
      int q = xb;
      while (q < xb + 16 && (sm.kc[q] & 7) == K_CONT) q++;
      int p = q - 1;
      while (p > q - 4 && (sm.kc[p] & 7) == K_CONT) p--;
      uint32_t cnt = 0;
      for (;;) {
        if (p < HALO) { reach_t0 = 1; break; }
        if ((sm.kc[p] & 7) != K_N || bit_get(sm.insp, p)) break;
        cnt++;
        if (bit_get(sm.pst, p)) break;
        if (cnt == NRUN_WALK) { unres = 1; break; }
        const int q2 = p;
        p--;
        while (p > q2 - 4 && (sm.kc[p] & 7) == K_CONT) p--;
      }
      r = cnt;
    }
    // the tile's carry (warp 0; thread 0 of every tile needs it)
    if (tid < 32) {
      int resolved = 0;
      uint32_t cnt = 0;
      if (tid == 0) {
        int p = HALO - 1;
        while (p > HALO - 5 && (sm.kc[p] & 7) == K_CONT) p--;
        for (;;) {
          if (p < TRUST) break;
          if ((sm.kc[p] & 7) != K_N || bit_get(sm.insp, p)) { resolved = 1; break; }
          cnt++;
          if (bit_get(sm.pst, p)) { resolved = 1; break; }
          const int q = p;
          p--;
          while (p > q - 5 && (sm.kc[p] & 7) == K_CONT) p--;
        }
      }
      resolved = __shfl_sync(0xffffffffu, resolved, 0);
      uint64_t carry;
      if (resolved) carry = cnt % 3;
      else carry = carry_walk_warp<NRunOp>(c.W.desc_a, tile, 0, c.W.status, 4);
      if (tid == 0) sm.ncarry = carry;
    }
    if (__syncthreads_or(unres)) {
      // a run of numbers longer than the walks: every thread's aggregate of
      // its 16 bytes, an inclusive warp scan, the warps before it
      uint32_t nreset = 0, ncount = 0;
      for (int j = 0; j < 16; j++) {
        const int x = xb + j;
        const uint8_t k = sm.kc[x] & 7;
        if (k == K_CONT) continue;
        if (k == K_OUT) break;
        if (k != K_N || bit_get(sm.insp, x)) { nreset = 1; ncount = 0; continue; }
        if (bit_get(sm.pst, x)) { nreset = 1; ncount = 0; }
        ncount = (ncount + 1) % 3;
      }
      const uint32_t mine = (nreset ? 0u : 4u) | ncount;
      uint32_t x = mine;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if ((tid & 31) >= o) x = (uint32_t)NRunOp::comb(y, x);
      }
      if ((tid & 31) == 31) sm.scan[tid >> 5] = x;
      __syncthreads();
      if (agg_late) {
        uint64_t agg = NRunOp::id();
        for (int w = 0; w < SPLIT_THREADS / 32; w++) agg = NRunOp::comb(agg, sm.scan[w]);
        st_relaxed_u64(&c.W.desc_a[tile], DESC_AGG | agg);
      }
      uint64_t pre = sm.ncarry;
      for (int w = 0; w < (tid >> 5); w++) pre = NRunOp::comb(pre, sm.scan[w]);
      uint32_t e = __shfl_up_sync(0xffffffffu, x, 1);
      if ((tid & 31) == 0) e = (uint32_t)NRunOp::id();
      r = (uint32_t)(NRunOp::comb(pre, e) & 3);
    } else if (reach_t0) {
      r += (uint32_t)(sm.ncarry & 3);
    }
    r %= 3u;
    // 6. the start test: 16 ASCII bytes at once where possible, else per code point
    {
      int ndef = 0;
      Win w{c, sm, wlo, 0, &ndef};
      uint32_t bits = 0;
      bool fast = wlo + xb + 20 <= c.n;
      uint32_t P[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t PS = 0;  // piece starts of bytes xb - 4 .. xb + 19
      if (fast) {
        const int b0 = xb - 4;
        const uint64_t ins = ((uint64_t)sm.insp[(b0 >> 5) + 1] << 32) | sm.insp[b0 >> 5];
        fast = ((ins >> (b0 & 31)) & 0xFFFFFFu) == 0;
        const uint64_t ps = ((uint64_t)sm.pst[(b0 >> 5) + 1] << 32) | sm.pst[b0 >> 5];
        PS = (uint32_t)(ps >> (b0 & 31)) & 0xFFFFFFu;
      }
      if (fast) {
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(&sm.kc[xb - 4]);
        const uint64_t y0 = transpose8x8(((uint64_t)kw[1] << 32) | kw[0]);
        const uint64_t y1 = transpose8x8(((uint64_t)kw[3] << 32) | kw[2]);
        const uint64_t y2 = transpose8x8(((uint64_t)kw[5] << 32) | kw[4]);
#pragma unroll
        for (int i = 0; i < 8; i++)
          P[i] = (uint32_t)((y0 >> (8 * i)) & 0xFFu) | ((uint32_t)((y1 >> (8 * i)) & 0xFFu) << 8) |
                 ((uint32_t)((y2 >> (8 * i)) & 0xFFu) << 16);
        fast = (P[1] & P[2] & 0xFFFFFFu) == 0;  // no continuation bytes or text end
      }
      if (fast) {
        uint32_t slow;
        bits = starts_ascii16(P, r, PS, &slow, c.T.pattern == TK_PATTERN_R50K_DIGITS);
        for (; slow; slow &= slow - 1) {
          const int j = __ffs(slow) - 1;
          w.owner = (tid << 4) | j;
          if (starts_here(w, wlo + xb + j, sm.kc[xb + j], 0)) bits |= 1u << j;
        }
      } else {
        for (int j = 0; j < 16; j++) {
          const int x = xb + j;
          const uint8_t k = sm.kc[x];
          const uint8_t k7 = k & 7;
          if (k7 == K_CONT) continue;
          if (k7 == K_OUT) break;
          const int64_t pos = wlo + x;
          uint32_t nidx = 0;
          const bool in_sp = bit_get(sm.insp, x);
          if (k7 == K_N && !in_sp) {
            if (bit_get(sm.pst, x)) r = 0;
            nidx = r;
            r = (r + 1) % 3;
          } else {
            r = 0;
          }
          bool s;
          if (in_sp) s = bit_get(sm.sst, x);
          else if (bit_get(sm.pst, x)) s = true;
          else {
            w.owner = (tid << 4) | j;
            s = starts_here(w, pos, k, nidx);
          }
          if (s) bits |= 1u << j;
        }
      }
      // deferred white-space walks: one warp each, then their start bits
      if (__syncthreads_or(ndef)) {
        const int nr = min(sm.nreq, WALK_MAX);
        for (int k = tid >> 5; k < nr; k += SPLIT_THREADS / 32) {
          const bool res = warp_ws_rest(c, sm.req_q[k], sm.req_check[k] != 0);
          if ((tid & 31) == 0) sm.req_res[k] = res ? 1 : 0;
        }
        __syncthreads();
        if (ndef)
          for (int k = 0; k < nr; k++)
            if ((sm.req_owner[k] >> 4) == tid && sm.req_res[k]) bits |= 1u << (sm.req_owner[k] & 15);
      }
      // 7. start bitmaps of the tile (two threads' 16 bits per word) and the
      //    position of its first start (tile_first starts at NO_START, set by
      //    k_reset).  No barrier after: the next tile writes shared memory
      //    only after the loop's first one.
      const uint32_t hi = __shfl_down_sync(0xffffffffu, bits, 1);
      if (!(tid & 1)) {
        const int64_t word = (t0 >> 5) + (tid >> 1);
        const uint32_t wv = bits | (hi << 16);
        c.W.pbits[word] = wv;
        if (c.T.n_spec) c.W.sbits[word] = wv & sm.sst[(HALO >> 5) + (tid >> 1)];
      }
      const uint32_t f = __reduce_min_sync(0xffffffffu, bits ? (uint32_t)(16 * tid + __ffs(bits) - 1) : 0xFFFFFFFFu);
      if ((tid & 31) == 0 && f != 0xFFFFFFFFu) atomicMin(&c.W.tile_first[tile], f);
    }
  }
}

// --------------------------------------------------------------------------
// Merging.  Pieces are token ids; the merged piece of a pair of rank r is the
// token r (rank = id), so the parts loop never touches bytes after its first
// round ("Inside encode: a parts vector and a linear scan").

// The same loop for a pre-token of n <= W bytes with every array in
// registers: fully unrolled, dynamic positions handled by predicated selects.
// b must have W readable bytes.
template <int W>
__device__ __forceinline__ int merge_reg(const MergeTabs T, const uint8_t* b, int n, int32_t* out) {
  static_assert(W <= 16, "positions are packed in four bits");
  // rk[i]: rank of the pair (i, i + 1), NOPAIR if none; ranks are below 2^20,
  // so (rank << 4 | i) orders by rank, then by position (the leftmost minimum)
  constexpr uint32_t NOPAIR = 0x0FFFFFFFu;
  uint32_t ids[W], rk[W];
#pragma unroll
  for (int i = 0; i < W; i++) {
    uint32_t v = 0;
    if (i < n) v = __ldg(&T.byte_id[b[i]]);
    ids[i] = v;
  }
#pragma unroll
  for (int i = 0; i < W - 1; i++) {
    uint32_t v = NOPAIR;
    if (i + 1 < n) {
      const uint32_t r = dense_rank(T, b[i], b[i + 1]);
      v = r == RANK_MAX ? NOPAIR : r;
    }
    rk[i] = v;
  }
  rk[W - 1] = NOPAIR;
  int m = n;
  while (m > 1) {
    uint32_t key = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < W - 1; i++) key = min(key, (rk[i] << 4) | (uint32_t)i);
    if (key >= (NOPAIR << 4)) break;
    const int bi = (int)(key & 15u);
    const uint32_t best = key >> 4;
    // piece bi becomes the token `best`; pieces after bi + 1 move down one
    uint32_t a_prev = 0, a_next = 0;
#pragma unroll
    for (int i = 0; i < W - 1; i++) {
      const bool gt = i > bi;
      const uint32_t nid = gt ? ids[i + 1] : (i == bi ? best : ids[i]);
      rk[i] = gt ? rk[i + 1] : rk[i];
      ids[i] = nid;
      a_prev = (i == bi - 1) ? nid : a_prev;
      a_next = (i == bi + 1) ? nid : a_next;
    }
    rk[W - 1] = NOPAIR;
    m--;
    // re-rank the pairs at bi and bi - 1
    uint32_t r0 = (bi + 1 < m) ? pair_rank(T, best, a_next) : RANK_MAX;
    uint32_t r1 = (bi > 0) ? pair_rank(T, a_prev, best) : RANK_MAX;
    r0 = r0 == RANK_MAX ? NOPAIR : r0;
    r1 = r1 == RANK_MAX ? NOPAIR : r1;
#pragma unroll
    for (int i = 0; i < W; i++) rk[i] = (i == bi) ? r0 : ((i == bi - 1) ? r1 : rk[i]);
  }
#pragma unroll
  for (int i = 0; i < W; i++)
    if (i < m) out[i] = (int32_t)ids[i];
  return m;
}

// Pre-tokens of 1..4 bytes, one code path for every length.  Every pair of
// adjacent parts spans a slice of the piece, so the loop only ever asks for
// the ranks of the byte pairs (dense table), the triples and the whole piece
// (slice table): loaded all at once (le4_load), then the loop written out by
// cases on the cut each round removes (le4_finish; cuts 1, 2, 3 between the
// bytes).  Positions past the piece's length take part in no slice, so they
// stay parts of their own at the end and are dropped from the result.
struct Le4 {
  int n;
  uint32_t w;               // the 4 bytes, little-endian
  uint32_t r01, r12, r23;   // byte pairs
  uint64_t sa, sb, sw;      // first probes of the slices 0-2, 1-3, 0-3 (~0: none)
};

__device__ __forceinline__ Le4 le4_load(const MergeTabs& T, const uint8_t* b, int n) {
  Le4 L;
  L.n = n;
  const uint32_t b0 = b[0], b1 = b[1], b2 = b[2], b3 = b[3];  // b has 4 readable bytes
  L.w = b0 | b1 << 8 | b2 << 16 | b3 << 24;
  L.sa = n > 2 ? s34_first(T, L.w & 0xFFFFFFu) : ~0ull;
  L.sb = n > 3 ? s34_first(T, L.w >> 8) : ~0ull;
  L.sw = n > 3 ? s34_first(T, L.w) : ~0ull;
  L.r01 = n > 1 ? dense_rank(T, b0, b1) : RANK_MAX;
  L.r12 = n > 2 ? dense_rank(T, b1, b2) : RANK_MAX;
  L.r23 = n > 3 ? dense_rank(T, b2, b3) : RANK_MAX;
  return L;
}

// Writes the piece's ids to out[0 .. count) and returns count (single-byte
// ids come from the 1 KB byte table here, after the slice loads).
__device__ __forceinline__ int le4_finish(const MergeTabs& T, const Le4& L, int32_t* out) {
  const uint32_t r012 = s34_rank(T, L.sa, L.w & 0xFFFFFFu, false), r123 = s34_rank(T, L.sb, L.w >> 8, false);
  const uint32_t r0123 = s34_rank(T, L.sw, L.w, true);
  const uint32_t r01 = L.r01, r12 = L.r12, r23 = L.r23;
  const uint32_t i0 = __ldg(&T.byte_id[L.w & 255u]), i1 = __ldg(&T.byte_id[(L.w >> 8) & 255u]);
  const uint32_t i2 = __ldg(&T.byte_id[(L.w >> 16) & 255u]), i3 = __ldg(&T.byte_id[L.w >> 24]);
  uint32_t p0, p1 = 0, p2 = 0, p3 = 0;
  int parts;
  if (r01 == RANK_MAX && r12 == RANK_MAX && r23 == RANK_MAX) {
    p0 = i0; p1 = i1; p2 = i2; p3 = i3;
    parts = 4;
  } else {
    // round 1 removes cut c1 (the leftmost least pair rank); round 2 sees
    //   c1 = 1: [01][2][3]  left slice 012, right slice 23
    //   c1 = 2: [0][12][3]  left slice 012, right slice 123
    //   c1 = 3: [0][1][23]  left slice 01,  right slice 123
    const int c1 = (r01 <= r12 && r01 <= r23) ? 1 : (r12 <= r23 ? 2 : 3);
    const uint32_t rl = c1 == 3 ? r01 : r012, rr = c1 == 1 ? r23 : r123;
    if (rl == RANK_MAX && rr == RANK_MAX) {
      p0 = c1 == 1 ? r01 : i0;
      p1 = c1 == 1 ? i2 : (c1 == 2 ? r12 : i1);
      p2 = c1 == 3 ? r23 : i3;
      parts = 3;
    } else if (r0123 != RANK_MAX) {  // round 3: the two parts left span the piece
      p0 = r0123;
      parts = 1;
    } else {
      //   left,  c1 != 3: [012][3];  left,  c1 == 3: [01][23]
      //   right, c1 == 1: [01][23];  right, c1 != 1: [0][123]
      const bool left = rl <= rr;
      const bool split22 = left ? c1 == 3 : c1 == 1;
      p0 = split22 ? r01 : (left ? r012 : i0);
      p1 = split22 ? r23 : (left ? i3 : r123);
      parts = 2;
    }
  }
  const int m = parts - (4 - L.n);
  out[0] = (int32_t)p0;
  if (m > 1) out[1] = (int32_t)p1;
  if (m > 2) out[2] = (int32_t)p2;
  if (m > 3) out[3] = (int32_t)p3;
  return m;
}

// The group that runs one round merge: NW warps (NW = 1: one warp, no block
// barriers; else the whole CTA).  s64 / s32 are shared scratch of NW entries.
template <int NW>
struct RGroup {
  static constexpr int kWarps = NW;
  int64_t* s64;
  uint32_t* s32;
  // the group's threads share one L1: plain loads see each other's stores
  template <class T>
  __device__ T ld(const T* p) const { return *p; }
  __device__ int warp() const { return NW == 1 ? 0 : (int)(threadIdx.x >> 5); }
  __device__ void sync() const {
    if (NW == 1) __syncwarp();
    else __syncthreads();
  }
  __device__ uint32_t gmin(uint32_t v) const {
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (NW == 1) return v;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s32[warp()] = v;
    __syncthreads();
    uint32_t r = s32[0];
    for (int k = 1; k < NW; k++) r = min(r, s32[k]);
    __syncthreads();
    return r;
  }
  // exclusive max (op 1) or sum (op 0) over the warps of one value per warp
  __device__ int64_t warp_excl(int64_t wv, int op, int64_t* total) const {
    const int64_t idv = op ? INT64_MIN : 0;
    if (NW == 1) {
      *total = wv;
      return idv;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s64[warp()] = wv;
    __syncthreads();
    int64_t e = idv, t = idv;
    for (int k = 0; k < NW; k++) {
      const int64_t v = s64[k];
      if (k < warp()) e = op ? max(e, v) : e + v;
      t = op ? max(t, v) : t + v;
    }
    __syncthreads();
    *total = t;
    return e;
  }
};

// Thread-block cluster primitives (inline PTX): rank in the cluster, the
// cluster-wide barrier (release / acquire at cluster scope), and loads from
// another CTA's shared memory.
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cl_ld32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ int64_t cl_ld64(uint32_t a) {
  int64_t v;
  asm volatile("ld.shared::cluster.s64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}

// The round-merge group of a whole cluster of CL CTAs of CW warps (one piece
// spread over CL SMs).  Reductions go through each CTA's shared memory and
// distributed shared memory; the merge buffers are read through L2 (.cg),
// since the CTAs sit on different SMs.  s64 / s32: 33 entries per CTA.
template <int CL, int CW>
struct CGroup {
  static_assert(CW >= 1 && CW <= 32, "warps per CTA");
  static constexpr int kWarps = CL * CW;
  int64_t* s64;
  uint32_t* s32;
  uint32_t rank;
  __device__ int warp() const { return (int)(rank * CW + (threadIdx.x >> 5)); }
  __device__ void sync() const { cl_sync(); }
  template <class T>
  __device__ T ld(const T* p) const { return __ldcg(p); }
  __device__ uint32_t gmin(uint32_t v) const {
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s32[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t u = threadIdx.x < CW ? s32[threadIdx.x] : 0xFFFFFFFFu;
      for (int o = 16; o > 0; o >>= 1) u = min(u, __shfl_xor_sync(0xffffffffu, u, o));
      if (threadIdx.x == 0) s32[32] = u;
    }
    cl_sync();
    uint32_t r = 0xFFFFFFFFu;
    for (int k = 0; k < CL; k++) r = min(r, cl_ld32(cl_map(&s32[32], (uint32_t)k)));
    cl_sync();
    return r;
  }
  __device__ int64_t warp_excl(int64_t wv, int op, int64_t* total) const {
    const int64_t idv = op ? INT64_MIN : 0;
    const int wl = (int)(threadIdx.x >> 5);
    if ((threadIdx.x & 31) == 0) s64[wl] = wv;
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t t = idv;
      for (int k = 0; k < CW; k++) t = op ? max(t, s64[k]) : t + s64[k];
      s64[32] = t;
    }
    cl_sync();
    int64_t e = idv, t = idv;
    for (int k = 0; k < wl; k++) e = op ? max(e, s64[k]) : e + s64[k];
    for (int r = 0; r < CL; r++) {
      const int64_t v = cl_ld64(cl_map(&s64[32], (uint32_t)r));
      if (r < (int)rank) e = op ? max(e, v) : e + v;
      t = op ? max(t, v) : t + v;
    }
    cl_sync();
    *total = t;
    return e;
  }
};

// Exact round merge of the pre-token text[s .. s+n) by a group (see the file
// header).  Each warp owns a contiguous chunk of the parts and its lanes take
// consecutive parts, so every pass reads and writes coalesced.  Works in the
// workspace at the piece's byte offset; the ids end in arena[s ..].  Returns
// the number of ids.
template <class Grp>
__device__ int64_t merge_rounds(const Call& c, const Grp& g, int64_t s, int64_t n) {
  constexpr int NW = Grp::kWarps;
  constexpr int U = 4;  // 32-element strips per batch: U loads in flight per lane
  const int64_t G = c.gb + s;
  uint32_t* A_ids = reinterpret_cast<uint32_t*>(c.W.arena + G);
  uint32_t* A_rk = c.W.lrk + G;
  uint32_t* B_ids = c.W.lids2 + G;
  uint32_t* B_rk = c.W.lrk2 + G;
  uint8_t* sel = c.W.lsel + G;
  uint8_t* chg = c.W.lchg + G;
  const int lane = threadIdx.x & 31, w = g.warp();
  const uint32_t lt = (1u << lane) - 1u;  // lanes below this one
  const int64_t n0 = n;
  for (int64_t i = (int64_t)w * 32 + lane; i < n; i += NW * 32) {
    const uint32_t b = gbyte(c, s + i);
    A_ids[i] = __ldg(&c.T.byte_id[b]);
    A_rk[i] = (i + 1 < n) ? __ldg(&c.T.dense[(b << 8) | gbyte(c, s + i + 1)]) : RANK_MAX;
  }
  g.sync();
  bool in_b = false;
  for (int64_t round = 0;; round++) {
    // each warp owns [wlo, whi): whole strips of 32, lanes on consecutive parts
    const int64_t cw = (((n + NW - 1) / NW) + 31) & ~(int64_t)31;
    const int64_t wlo = min(n, (int64_t)w * cw), whi = min(n, wlo + cw);
    // (1) the minimum pair rank
    uint32_t m = RANK_MAX;
    for (int64_t b0 = wlo; b0 < whi; b0 += 32 * U) {
      uint32_t v[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        v[u] = i < whi ? g.ld(&A_rk[i]) : RANK_MAX;
      }
#pragma unroll
      for (int u = 0; u < U; u++) m = min(m, v[u]);
    }
    const uint32_t rs = g.gmin(m);
    if (rs == RANK_MAX) break;
    // (2) chains of rs-pairs: every other pair from each chain's start.  The
    //     last non-candidate before each part comes from ballots and a carry.
    int64_t ln_w = -1;
    for (int64_t b0 = wlo; b0 < whi; b0 += 32 * U) {
      uint32_t v[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        v[u] = i < whi ? g.ld(&A_rk[i]) : rs;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const uint32_t nm = __ballot_sync(0xffffffffu, v[u] != rs);
        if (nm) ln_w = b0 + 32 * u + 31 - __clz(nm);
      }
    }
    int64_t tot;
    int64_t carry = g.warp_excl(ln_w, 1, &tot);
    if (carry < -1) carry = -1;
    for (int64_t b0 = wlo; b0 < whi; b0 += 32 * U) {
      uint32_t v[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        v[u] = i < whi ? g.ld(&A_rk[i]) : rs;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t b = b0 + 32 * u, i = b + lane;
        const bool in = i < whi;
        const bool cand = in && v[u] == rs;
        const uint32_t nm = __ballot_sync(0xffffffffu, in && !cand);
        const uint32_t before = nm & lt;
        const int64_t ln = before ? b + 31 - __clz(before) : carry;
        if (in) sel[i] = cand && (((i - ln - 1) & 1) == 0);
        if (nm) carry = b + 31 - __clz(nm);
      }
    }
    g.sync();
    // (3) the first selected merge that creates a neighbour pair of lower rank
    //     (only possible when the token rs has an extension ranked below it)
    const uint32_t xf = __ldg(&c.T.ext_low[rs]);
    uint32_t fb = 0xFFFFFFFFu;
    for (int64_t b0 = wlo; xf && b0 < whi && fb == 0xFFFFFFFFu; b0 += 32 * U) {
      uint8_t sv[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        sv[u] = i < whi ? g.ld(&sel[i]) : 0;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        bool bad = false;
        if (sv[u]) {
          const uint32_t left = i >= 1 ? ((i >= 2 && g.ld(&sel[i - 2])) ? rs : g.ld(&A_ids[i - 1])) : 0u;
          const uint32_t right = i + 2 < n ? g.ld(&A_ids[i + 2]) : 0u;
          const uint32_t rl = i >= 1 ? pair_rank(c.T, left, rs) : RANK_MAX;
          const uint32_t rr = i + 2 < n ? pair_rank(c.T, rs, right) : RANK_MAX;
          bad = rl < rs || rr < rs;
        }
        const uint32_t bm = __ballot_sync(0xffffffffu, bad);
        if (bm && fb == 0xFFFFFFFFu) fb = (uint32_t)(b0 + 32 * u + __ffs(bm) - 1);
      }
    }
    const uint32_t limit = xf ? g.gmin(fb) : 0xFFFFFFFFu;
    // (4) merge the selected pairs up to limit, compacting into B
    int64_t keep_w = 0;
    for (int64_t b0 = wlo; b0 < whi; b0 += 32 * U) {
      uint8_t pv[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        pv[u] = (i < whi && i >= 1) ? g.ld(&sel[i - 1]) : 0;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        const bool kp = i < whi && !(pv[u] && (uint64_t)(i - 1) <= (uint64_t)limit);
        keep_w += __popc(__ballot_sync(0xffffffffu, kp));
      }
    }
    int64_t dst = g.warp_excl(keep_w, 0, &tot);
    const int64_t n2 = tot;
    for (int64_t b0 = wlo; b0 < whi; b0 += 32 * U) {
      uint8_t pv[U], sv[U];
      uint32_t iv[U], rv[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        const bool in = i < whi;
        pv[u] = (in && i >= 1) ? g.ld(&sel[i - 1]) : 0;
        sv[u] = in ? g.ld(&sel[i]) : 0;
        iv[u] = in ? g.ld(&A_ids[i]) : 0u;
        rv[u] = in ? g.ld(&A_rk[i]) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t i = b0 + 32 * u + lane;
        const bool kp = i < whi && !(pv[u] && (uint64_t)(i - 1) <= (uint64_t)limit);
        const uint32_t km = __ballot_sync(0xffffffffu, kp);
        if (kp) {
          const int64_t pos = dst + __popc(km & lt);
          const bool merged = sv[u] && (uint64_t)i <= (uint64_t)limit;
          B_ids[pos] = merged ? rs : iv[u];
          B_rk[pos] = rv[u];
          chg[pos] = merged;
        }
        dst += __popc(km);
      }
    }
    g.sync();
    // (5) re-rank the pairs next to merged pieces
    for (int64_t q0 = (int64_t)w * 32; q0 < n2; q0 += (int64_t)NW * 32 * U) {
      uint8_t c0[U], c1[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t q = q0 + (int64_t)NW * 32 * u + lane;
        c0[u] = q < n2 ? g.ld(&chg[q]) : 0;
        c1[u] = q + 1 < n2 ? g.ld(&chg[q + 1]) : 0;
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int64_t q = q0 + (int64_t)NW * 32 * u + lane;
        if (q + 1 == n2) B_rk[q] = RANK_MAX;
        else if (q + 1 < n2 && (c0[u] || c1[u])) B_rk[q] = pair_rank(c.T, g.ld(&B_ids[q]), g.ld(&B_ids[q + 1]));
      }
    }
    g.sync();
    uint32_t* t1 = A_ids; A_ids = B_ids; B_ids = t1;
    uint32_t* t2 = A_rk; A_rk = B_rk; B_rk = t2;
    in_b = !in_b;
    n = n2;
    // every round merges at least one pair, so n0 rounds always suffice
    if (round > n0) {
      if (threadIdx.x == 0) set_error(c.W.status, TK_E_LIMIT, 6);
      break;
    }
  }
  if (in_b) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(c.W.arena + G);
    for (int64_t i = (int64_t)w * 32 + lane; i < n; i += NW * 32) dst[i] = g.ld(&A_ids[i]);
    g.sync();
  }
  return n;
}

// The same rounds over warp-owned chunks, for one CTA of NW warps.  Warp w
// owns chunk w: its parts sit at the front of a fixed window of cw slots, in
// text order, and the pair rank of a part is the rank with the next part in
// text order (the first part of the next non-empty chunk for the last one).
// A round merges every other pair of rank rs from the start of each run of
// rs-pairs, up to the first merge that creates a lower-ranked neighbour pair,
// as above; but each chunk compacts in place (no scan over the CTA), and the
// chunks without an rs-pair (most of them, in the late rounds of a long
// piece, which merge a few pairs each) do nothing but keep their minimum
// rank.  A run of rs-pairs entering a chunk from the chunks before it flips
// the choices in the chunk's leading run when its length there is odd.
// Works in the workspace at the piece's byte offset until the parts fit in
// the CTA's shared memory `sm` (scap parts, CHUNK_PART bytes each), then
// there; the ids end in arena[s ..].  Returns the number of ids.
constexpr int CHUNK_PART = 9;  // id and rank (4 + 4 bytes), chosen / merged flag
template <int NW>
struct ChunkSh {
  int cnt[NW], cnt2[NW];   // parts in each chunk (at the round's start / after it)
  uint32_t mn[NW];         // each chunk's minimum pair rank
  int lead[NW], tail[NW];  // the chunk's rs-pairs before its first / after its last other pair
  uint32_t bad[NW];        // the chunk's first merge that stops the round
  int off[NW + 1];         // chunk offsets in text order
};

// The part d places after (d > 0) or before (d < 0) part j of chunk w, in
// text order over the non-empty chunks; false if there is none.
template <int NW>
__device__ __forceinline__ bool chunk_step(const int* cnt, int& w, int& j, int d) {
  for (; d > 0; d--) {
    if (j + 1 < cnt[w]) { j++; continue; }
    int v = w + 1;
    while (v < NW && cnt[v] == 0) v++;
    if (v >= NW) return false;
    w = v; j = 0;
  }
  for (; d < 0; d++) {
    if (j > 0) { j--; continue; }
    int v = w - 1;
    while (v >= 0 && cnt[v] == 0) v--;
    if (v < 0) return false;
    w = v; j = cnt[v] - 1;
  }
  return true;
}

template <int NW>
__device__ int64_t merge_chunks(const Call& c, int64_t s, int64_t n, uint8_t* sm, int64_t scap, ChunkSh<NW>& S) {
  constexpr int U = 4;
  constexpr uint32_t NONE = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31, w = (int)(threadIdx.x >> 5);
  const uint32_t lt = (1u << lane) - 1u;
  const int64_t G = c.gb + s;
  uint32_t* const out = reinterpret_cast<uint32_t*>(c.W.arena + G);
  bool on_chip = scap > 0 && n <= scap;
  uint32_t* ids = on_chip ? reinterpret_cast<uint32_t*>(sm) : c.W.lids2 + G;
  uint32_t* rk = on_chip ? ids + scap : c.W.lrk + G;
  uint8_t* sel = on_chip ? reinterpret_cast<uint8_t*>(rk + scap) : c.W.lsel + G;
  int cw = (int)((((n + NW - 1) / NW) + 31) & ~(int64_t)31);
  // the chunk's minimum pair rank and its pairs of that rank before the first
  // and after the last other pair, into S.mn / S.lead / S.tail
  auto chunk_stats = [&](int cnt) {
    uint32_t m = RANK_MAX;
    for (int j = lane; j < cnt; j += 32) m = min(m, rk[w * cw + j]);
    m = __reduce_min_sync(0xffffffffu, m);
    int first = cnt, last = -1;
    if (m != RANK_MAX) {
      for (int b0 = 0; b0 < cnt; b0 += 32) {
        const int j = b0 + lane;
        const uint32_t ne = __ballot_sync(0xffffffffu, j < cnt && rk[w * cw + j] != m);
        if (ne) {
          if (first == cnt) first = b0 + __ffs(ne) - 1;
          last = b0 + 31 - __clz(ne);
        }
      }
    }
    if (lane == 0) {
      S.mn[w] = m;
      S.lead[w] = first;
      S.tail[w] = cnt - 1 - last;
    }
  };
  // length of the run of rs-pairs that ends just before chunk v (rs: the
  // minimum of every chunk it crosses; empty chunks are transparent)
  auto run_into = [&](int v, uint32_t rs) {
    int r = 0;
    for (int u = v - 1; u >= 0; u--) {
      if (S.cnt[u] == 0) continue;
      if (S.mn[u] != rs) break;
      r += S.tail[u];
      if (S.lead[u] != S.cnt[u]) break;
    }
    return r;
  };
  {
    const int cnt = (int)max((int64_t)0, min((int64_t)cw, n - (int64_t)w * cw));
    for (int j = lane; j < cnt; j += 32) {
      const int64_t i = (int64_t)w * cw + j;
      const uint32_t b = gbyte(c, s + i);
      ids[w * cw + j] = __ldg(&c.T.byte_id[b]);
      rk[w * cw + j] = (i + 1 < n) ? __ldg(&c.T.dense[(b << 8) | gbyte(c, s + i + 1)]) : RANK_MAX;
    }
    __syncwarp();
    chunk_stats(cnt);
    if (lane == 0) S.cnt[w] = cnt;
  }
  __syncthreads();
  for (int64_t round = 0;; round++) {
    static_assert(NW <= 32, "one chunk minimum per lane");
    const uint32_t rs = __reduce_min_sync(0xffffffffu, lane < NW ? S.mn[lane] : RANK_MAX);
    if (rs == RANK_MAX) break;
    const int cnt = S.cnt[w];
    const bool act = S.mn[w] == rs;
    const int base = w * cw;
    // Only a token rs with an extension that ranks below it can stop a round
    // early; without one, a round chooses and merges in one pass per chunk.
    const uint32_t xf = __ldg(&c.T.ext_low[rs]);
    bool moves = act;
    int cnt2 = cnt;
    if (!xf) {
      // whether the chunk's first part is taken by the last pair before it:
      // that pair is an rs-pair at an even place in its run
      bool first_gone = false;
      if (cnt > 0) {
        int v = w - 1;
        while (v >= 0 && S.cnt[v] == 0) v--;
        if (v >= 0 && S.mn[v] == rs && S.tail[v] > 0) {
          const int at = (S.lead[v] == S.cnt[v] ? run_into(v, rs) : 0) + S.tail[v] - 1;
          first_gone = (at & 1) == 0;
        }
      }
      moves = act || first_gone;
      if (moves) {
        // choose every other rs-pair of each run (counting the run entering
        // the chunk) and compact in place, the merged flags into sel
        int carry = -1 - (act && S.lead[w] > 0 ? run_into(w, rs) : 0);
        int dst = 0;
        bool prev = first_gone;  // chosen flag of the pair before the strip's lane 0
        for (int b0 = 0; b0 < cnt; b0 += 32 * U) {
          uint32_t iv[U], rv[U];
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            const bool in = j < cnt;
            iv[u] = in ? ids[base + j] : 0u;
            rv[u] = in ? rk[base + j] : 0u;
          }
          __syncwarp();
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int b = b0 + 32 * u, j = b + lane;
            const bool in = j < cnt, cand = in && rv[u] == rs;
            const uint32_t nm = __ballot_sync(0xffffffffu, in && !cand);
            const uint32_t before = nm & lt;
            const int ln = before ? b + 31 - __clz(before) : carry;
            const bool chosen = cand && (((j - ln - 1) & 1) == 0);
            const bool up = __shfl_up_sync(0xffffffffu, (uint32_t)chosen, 1) != 0;
            const bool gone = lane == 0 ? prev : up;  // taken into the pair before it
            const bool kp = in && !gone;
            const uint32_t km = __ballot_sync(0xffffffffu, kp);
            if (kp) {
              const int pos = dst + __popc(km & lt);
              ids[base + pos] = chosen ? rs : iv[u];
              rk[base + pos] = rv[u];
              sel[base + pos] = chosen;
            }
            dst += __popc(km);
            prev = __shfl_sync(0xffffffffu, (uint32_t)chosen, 31) != 0;
            if (nm) carry = b + 31 - __clz(nm);
          }
          __syncwarp();
        }
        cnt2 = dst;
      }
    } else {
      // (1) choose every other rs-pair from the start of each run, counting
      //     runs as if they started in this chunk
      if (act) {
        int carry = -1, first_nc = cnt;
        for (int b0 = 0; b0 < cnt; b0 += 32 * U) {
          uint32_t v[U];
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            v[u] = j < cnt ? rk[base + j] : rs;
          }
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int b = b0 + 32 * u, j = b + lane;
            const bool in = j < cnt, cand = in && v[u] == rs;
            const uint32_t nm = __ballot_sync(0xffffffffu, in && !cand);
            const uint32_t before = nm & lt;
            const int ln = before ? b + 31 - __clz(before) : carry;
            if (in) sel[base + j] = cand && (((j - ln - 1) & 1) == 0);
            if (nm) {
              if (first_nc == cnt) first_nc = b + __ffs(nm) - 1;
              carry = b + 31 - __clz(nm);
            }
          }
        }
        if (lane == 0) {
          S.lead[w] = first_nc;
          S.tail[w] = cnt - 1 - carry;
        }
      }
      __syncthreads();
      // (2) a run entering the chunk with an odd length flips its leading run
      if (act && S.lead[w] > 0) {
        const int run_in = run_into(w, rs);
        if (run_in & 1) {
          __syncwarp();
          for (int j = lane; j < S.lead[w]; j += 32) sel[base + j] ^= 1;
        }
      }
      __syncthreads();
      // (3) the chunk's first chosen merge that creates a neighbour pair of a
      //     rank below rs (the one-at-a-time loop would take that pair next);
      //     the neighbours' first probes of a batch are loaded together
      int lw = NW;
      uint32_t lj = 0;
      if (act) {
        uint32_t fb = NONE;
        for (int b0 = 0; b0 < cnt && fb == NONE; b0 += 32 * U) {
          uint8_t sv[U];
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            sv[u] = j < cnt ? sel[base + j] : 0;
          }
          PairProbe pl[U], pq[U];
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            uint32_t left = 0, right = 0;
            bool hl = false, hr = false;
            if (sv[u]) {
              // the part before j, or rs when the pair before that one is chosen
              // (it merges first); the part two after j
              if (j >= 2) {
                hl = true;
                left = sel[base + j - 2] ? rs : ids[base + j - 1];
              } else {
                int pw = w, pj = j;
                if (chunk_step<NW>(S.cnt, pw, pj, -1)) {
                  int qw = pw, qj = pj;
                  const bool ql = chunk_step<NW>(S.cnt, qw, qj, -1) && S.mn[qw] == rs && sel[qw * cw + qj];
                  hl = true;
                  left = ql ? rs : ids[pw * cw + pj];
                }
              }
              if (j + 2 < cnt) {
                hr = true;
                right = ids[base + j + 2];
              } else {
                int qw = w, qj = j;
                if (chunk_step<NW>(S.cnt, qw, qj, 2)) {
                  hr = true;
                  right = ids[qw * cw + qj];
                }
              }
            }
            pl[u] = pair_first(c.T, left, rs, hl);
            pq[u] = pair_first(c.T, rs, right, hr);
          }
#pragma unroll
          for (int u = 0; u < U; u++) {
            const bool bad = sv[u] && (pair_finish(c.T, pl[u]) < rs || pair_finish(c.T, pq[u]) < rs);
            const uint32_t bm = __ballot_sync(0xffffffffu, bad);
            if (bm && fb == NONE) fb = (uint32_t)(b0 + 32 * u + __ffs(bm) - 1);
          }
        }
        if (lane == 0) S.bad[w] = fb;
      }
      // the round's limit: merges at (chunk, index) <= (lw, lj) go ahead
      __syncthreads();
      for (int k = 0; k < NW; k++)
        if (S.mn[k] == rs && S.bad[k] != NONE) {
          lw = k;
          lj = S.bad[k];
          break;
        }
      auto allowed = [&](int v, int j) { return v < lw || (v == lw && (uint32_t)j <= lj); };
      // (4) merge: each chunk compacts in place, the merged flags replacing
      //     the chosen ones in sel.  A chunk changes when it holds a chosen
      //     merge or its first part is taken by the chunk before it.
      bool first_gone = false;
      if (cnt > 0) {
        int pw = w, pj = 0;
        if (chunk_step<NW>(S.cnt, pw, pj, -1))
          first_gone = S.mn[pw] == rs && sel[pw * cw + pj] && allowed(pw, pj);
      }
      __syncthreads();  // every chunk's last chosen flag is read
      moves = act || first_gone;
      if (moves) {
        int dst = 0;
        uint8_t prev = first_gone ? 1 : 0;  // chosen flag of the pair before the strip's lane 0
        for (int b0 = 0; b0 < cnt; b0 += 32 * U) {
          uint32_t iv[U], rv[U];
          uint8_t sv[U];
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            const bool in = j < cnt;
            iv[u] = in ? ids[base + j] : 0u;
            rv[u] = in ? rk[base + j] : 0u;
            sv[u] = (in && act) ? sel[base + j] : 0;
          }
          __syncwarp();
#pragma unroll
          for (int u = 0; u < U; u++) {
            const int j = b0 + 32 * u + lane;
            const bool in = j < cnt;
            // the pair before part j merged: part j is taken into it
            const uint8_t up = (uint8_t)__shfl_up_sync(0xffffffffu, (uint32_t)sv[u], 1);
            const bool gone = lane == 0 ? (j == 0 ? first_gone : (prev && allowed(w, j - 1)))
                                        : (up && allowed(w, j - 1));
            const bool kp = in && !gone;
            const uint32_t km = __ballot_sync(0xffffffffu, kp);
            if (kp) {
              const int pos = dst + __popc(km & lt);
              const bool merged = sv[u] && allowed(w, j);
              ids[base + pos] = merged ? rs : iv[u];
              rk[base + pos] = rv[u];
              sel[base + pos] = merged;
            }
            dst += __popc(km);
            prev = (uint8_t)__shfl_sync(0xffffffffu, (uint32_t)sv[u], 31);
          }
          __syncwarp();
        }
        cnt2 = dst;
      }
    }
    if (lane == 0) S.cnt2[w] = cnt2;
    __syncthreads();
    // (5) re-rank the pairs of merged parts and of the parts before them
    //     (first probes of a batch loaded together)
    if (moves) {
      for (int j0 = 0; j0 < cnt2; j0 += 32 * U) {
        bool mg[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
          const int j = j0 + 32 * u + lane;
          mg[u] = j < cnt2 && sel[base + j];
        }
        PairProbe pn[U], pp[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
          const int j = j0 + 32 * u + lane;
          uint32_t x = 0, nxt = 0, prv = 0;
          bool hn = false, hp = false;
          if (mg[u]) {
            x = ids[base + j];
            int qw = w, qj = j;
            if (chunk_step<NW>(S.cnt2, qw, qj, 1)) {
              hn = true;
              nxt = ids[qw * cw + qj];
            }
            int pw = w, pj = j;
            if (chunk_step<NW>(S.cnt2, pw, pj, -1)) {
              hp = true;
              prv = ids[pw * cw + pj];
            }
          }
          pn[u] = pair_first(c.T, x, nxt, hn);  // unused probes resolve to RANK_MAX
          pp[u] = pair_first(c.T, prv, x, hp);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
          if (!mg[u]) continue;
          const int j = j0 + 32 * u + lane;
          rk[base + j] = pair_finish(c.T, pn[u]);
          int pw = w, pj = j;
          if (chunk_step<NW>(S.cnt2, pw, pj, -1)) rk[pw * cw + pj] = pair_finish(c.T, pp[u]);
        }
      }
    }
    __syncthreads();
    // (6) new minima: the chunks that moved and the non-empty chunk before each
    //     (only a chunk with a chosen pair writes ranks: its merged parts')
    bool dirty = moves;
    if (!dirty && cnt2 > 0) {
      for (int v = w + 1; v < NW; v++) {
        if (S.cnt2[v] == 0) continue;
        dirty = S.mn[v] == rs;
        break;
      }
    }
    __syncthreads();  // every warp has read the old minima and counts
    if (dirty) chunk_stats(cnt2);
    if (lane == 0) S.cnt[w] = cnt2;
    if (round > n) {  // every round merges at least one pair
      if (threadIdx.x == 0) set_error(c.W.status, TK_E_LIMIT, 6);
      __syncthreads();
      break;
    }
    __syncthreads();
    // once the parts fit, the rest of the rounds run in shared memory
    if (!on_chip && scap > 0) {
      if (threadIdx.x == 0) {
        int t = 0;
        for (int k = 0; k < NW; k++) {
          S.off[k] = t;
          t += S.cnt[k];
        }
        S.off[NW] = t;
      }
      __syncthreads();
      const int tot = S.off[NW];
      if (tot <= scap) {
        uint32_t* ids2 = reinterpret_cast<uint32_t*>(sm);
        uint32_t* rk2 = ids2 + scap;
        const int c0 = S.cnt[w], o0 = S.off[w];
        for (int j = lane; j < c0; j += 32) {
          ids2[o0 + j] = ids[base + j];
          rk2[o0 + j] = rk[base + j];
        }
        on_chip = true;
        ids = ids2;
        rk = rk2;
        sel = reinterpret_cast<uint8_t*>(rk + scap);
        cw = (((tot + NW - 1) / NW) + 31) & ~31;
        __syncthreads();
        const int cn = max(0, min(cw, tot - w * cw));
        chunk_stats(cn);
        if (lane == 0) S.cnt[w] = cn;
        __syncthreads();
      }
    }
  }
  // the chunks in text order to arena[s ..]
  if (threadIdx.x == 0) {
    int t = 0;
    for (int k = 0; k < NW; k++) {
      S.off[k] = t;
      t += S.cnt[k];
    }
    S.off[NW] = t;
  }
  __syncthreads();
  {
    const int c0 = S.cnt[w], o0 = S.off[w];
    for (int j = lane; j < c0; j += 32) out[o0 + j] = ids[w * cw + j];
  }
  const int64_t total = S.off[NW];
  __syncthreads();
  return total;
}

// --------------------------------------------------------------------------
// Fused encode of one 4 KiB tile: the pre-tokens of up to MID_MIN - 1 bytes
// that start in the tile are merged here (one thread each), their ids
// compacted in shared memory and staged with the tile's count.  Longer ones
// (merged by k_merge_mid and the long-piece kernels, on the side stream) are
// entries of the slot's table, in text order, for k_long_fixup.

constexpr int ETHREADS = 256;
constexpr int MERGE_U = 2;  // short pieces per thread per merge round
constexpr int EPAD = 96;                 // bytes loaded past the tile (short pieces, specials)
constexpr int MEDIUM_MAX = 1024;
constexpr int64_t CLUSTER_MIN = 32768;   // longer pieces merge on a CTA cluster
constexpr int MERGE_CL = 8;              // CTAs per cluster (portable size)
constexpr int MAX_GP = TILE / MID_MIN + 2;  // table entries of a tile (pieces of >= MID_MIN bytes)
constexpr uint32_t NO_START = 0xFFFFFFFFu;
// Staging slot per tile (u32 entries): the short ids from the front (rounded
// up to 4), 4 words per table entry from the back.  Pieces starting in the
// tile are disjoint and the table's are at least MID_MIN bytes long, so the
// short ids + MID_MIN * entries <= TILE + MID_MIN - 1: both parts fit.
constexpr int64_t STG = TILE + SHORT_MAX + 8;
static_assert(MID_MIN >= 5 && TILE + MID_MIN - 1 + 3 <= STG, "staging slot bound");
constexpr uint32_t DTAB_LOG2 = 20;                  // dedup table of long pieces: 2^20 slots

constexpr int LIST_END = TILE + SHORT_MAX;  // the mid pieces' list ends here
struct EncSmem {
  uint8_t text[TILE + EPAD + 16];
  uint32_t pb[(TILE + EPAD) / 32 + 1];  // pre-token starts in [t0, t0 + TILE + EPAD)
  uint32_t sb[TILE / 32];               // special starts
  uint32_t gb[TILE / 32];               // starts of pieces merged through global memory
  uint8_t cnt[TILE];                    // ids of the short piece starting at each byte
  int32_t stage[TILE + SHORT_MAX];      // ids of short pieces, at their start byte
  union {
    uint16_t list[TILE + SHORT_MAX];    // work lists: x | (len - 1) << 12 (until the merges end):
                                        // 3-4-byte pieces from the front, mid pieces from the back
    __align__(16) int32_t outs[TILE + SHORT_MAX + 4];  // then the tile's short ids in order
  };
  uint32_t th_full[ETHREADS];           // short ids before each thread's 16 bytes
  uint16_t th_gp[ETHREADS];             // table entries before each thread's 16 bytes
  uint32_t warp_tot[2 * ETHREADS / 32];
  int n_gp;
  uint32_t n_starts;
  uint32_t tile_short;
  int64_t seg[2];
};

__device__ int32_t special_id_smem(const Tables& T, const uint8_t* b, int len) {
  for (int k = 0; k < T.n_spec; k++) {
    const int L = T.spec_off[k + 1] - T.spec_off[k];
    if (L != len) continue;
    bool m = true;
    for (int j = 0; j < L && m; j++) m = b[j] == T.spec_bytes[T.spec_off[k] + j];
    if (m) return T.spec_ids[k];
  }
  return -1;
}

// Short ids before byte x of the tile (x in [0, TILE)), counted from the tile
// start, | the table entries before x << 16 (k_long_fixup replaces them by
// the ids of those entries).
__device__ uint32_t ids_before(const EncSmem& sm, int x) {
  const int t = x >> 4;
  uint32_t r = sm.th_full[t], g = sm.th_gp[t];
  for (int y = t << 4; y < x; y++) {
    if (!((sm.pb[y >> 5] >> (y & 31)) & 1u)) continue;  // not a pre-token start
    if (!((sm.gb[y >> 5] >> (y & 31)) & 1u)) r += sm.cnt[y];
    else g++;
  }
  return r | (g << 16);
}

template <bool MIDS>
__global__ void __launch_bounds__(ETHREADS, 5) k_encode_tiles(Call c) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  EncSmem& sm = *reinterpret_cast<EncSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const bool aligned = ((uintptr_t)c.text & 15) == 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t0 = tile * TILE;
    // 1. bytes, start bits (positions >= n read as no start), special starts
    for (int v = tid; v < (TILE + EPAD + 16) / 16; v += ETHREADS) {
      const int64_t p = t0 + 16 * v;
      if (aligned && p + 16 <= c.n) {
        *reinterpret_cast<uint4*>(&sm.text[16 * v]) = ld_na_v4(c.text + p);
      } else {
        for (int j = 0; j < 16; j++) sm.text[16 * v + j] = gbyte(c, p + j);
      }
    }
    for (int i = tid; i < (TILE + EPAD) / 32 + 1; i += ETHREADS) {
      const int64_t p = t0 + 32 * i;
      uint32_t w = 0;
      if (p < c.n) {
        w = c.W.pbits[(t0 >> 5) + i];
        if (p + 32 > c.n) w &= (1u << (c.n - p)) - 1u;
      }
      sm.pb[i] = w;
    }
    for (int i = tid; i < TILE / 32; i += ETHREADS) {
      sm.sb[i] = c.T.n_spec ? c.W.sbits[(t0 >> 5) + i] : 0u;
      sm.gb[i] = 0;
    }
    if (tid == 0) {
      sm.n_starts = 0;
      sm.seg[0] = c.W.tile_segs[4 * tile + 1];
      sm.seg[1] = (tile == ntiles - 1) ? c.S + 1 : c.W.tile_segs[4 * tile + 2];
    }
    __syncthreads();
    // 2. each thread: its pre-tokens (starts in bytes [16 tid, 16 tid + 16))
    const int xb = tid * 16;
    const uint32_t my = (sm.pb[xb >> 5] >> (xb & 31)) & 0xFFFFu;
    // 2a. lengths, as bit masks over a 48-bit window of the start bitmap (a
    //     virtual start at the text end): a start whose next start is k bytes
    //     on begins a piece of k bytes.  Pieces of one byte are their id, of
    //     two bytes the dense pair table or the two byte ids; pieces of three
    //     or four bytes are listed for the merge below; longer ones are
    //     flagged for the side streams' merges; specials (their exact end
    //     found one by one) are their id.
    uint64_t win = (((uint64_t)sm.pb[(xb >> 5) + 1] << 32) | sm.pb[xb >> 5]) >> (xb & 31);
    {
      const int64_t e = c.n - (t0 + xb);
      if (e >= 0 && e < 48) win |= 1ull << e;
    }
    const uint32_t n1 = (uint32_t)(win >> 1), n2 = (uint32_t)(win >> 2), n3 = (uint32_t)(win >> 3),
                   n4 = (uint32_t)(win >> 4);
    const uint32_t spc = my & ((sm.sb[xb >> 5] >> (xb & 31)) & 0xFFFFu);
    const uint32_t ord = my & ~spc;
    const uint32_t m1 = ord & n1, m2 = ord & ~n1 & n2, m3 = ord & ~n1 & ~n2 & n3;
    const uint32_t m4 = ord & ~n1 & ~n2 & ~n3 & n4, mg = ord & ~(n1 | n2 | n3 | n4);
    uint32_t inl = (uint32_t)__popc(m1 | spc);  // short ids of the pieces resolved here
    for (uint32_t bits = m1; bits; bits &= bits - 1) {
      const int x = xb + __ffs(bits) - 1;
      sm.stage[x] = (int32_t)__ldg(&c.T.byte_id[sm.text[x]]);
      sm.cnt[x] = 1;
    }
    for (uint32_t bits = m2; bits; bits &= bits - 1) {
      const int x = xb + __ffs(bits) - 1;
      const uint32_t b0 = sm.text[x], b1 = sm.text[x + 1];
      const uint32_t r = __ldg(&c.T.dense[(b0 << 8) | b1]);
      if (r != RANK_MAX) {
        sm.stage[x] = (int32_t)r;
        sm.cnt[x] = 1;
        inl += 1;
      } else {
        sm.stage[x] = (int32_t)__ldg(&c.T.byte_id[b0]);
        sm.stage[x + 1] = (int32_t)__ldg(&c.T.byte_id[b1]);
        sm.cnt[x] = 2;
        inl += 2;
      }
    }
    for (uint32_t bits = spc; bits; bits &= bits - 1) {
      const int x = xb + __ffs(bits) - 1;
      // a special: its exact end (the next start bit, else the first start
      // of a later tile, else n)
      int64_t e = -1;
      int y = x + 1;
      while (y < TILE + EPAD) {
        const uint32_t w = sm.pb[y >> 5] >> (y & 31);
        if (w) { y += __ffs(w) - 1; break; }
        y = (y | 31) + 1;
      }
      if (y < TILE + EPAD) e = t0 + y;
      else if (t0 + TILE + EPAD >= c.n) e = c.n;
      else {
        for (int64_t k = tile + 1; k < ntiles && e < 0; k++) {
          const uint32_t f = c.W.tile_first[k];
          if (f != NO_START) e = k * TILE + f;
        }
        if (e < 0) e = c.n;
      }
      sm.stage[x] = special_id_smem(c.T, &sm.text[x], (int)(e - (t0 + x)));
      sm.cnt[x] = 1;
    }
    // with MIDS, pieces of 5..SHORT_MAX bytes (the next start within 16
    // bytes) are merged here too, after the short ones; longer pieces (and
    // without MIDS the mid pieces) are merged on the side streams, which may
    // still be running: the tile records where they are, k_long_fixup adds
    // their ids' count
    uint32_t mid = 0, mlen = 0;  // mid pieces; their lengths - 1, 4 bits each, in start order
    for (uint32_t bits = MIDS ? mg : 0u; bits; bits &= bits - 1) {
      const int j = __ffs(bits) - 1;
      const uint32_t nx = (uint32_t)(win >> (j + 1)) & 0xFFFFu;
      if (nx) {
        mid |= 1u << j;
        mlen = (mlen >> 4) | ((uint32_t)(__ffs(nx) - 1) << 28);
      }
    }
    const uint32_t lng = mg & ~mid;
    if (lng) atomicOr(&sm.gb[xb >> 5], lng << (xb & 31));
    const uint32_t lst = m3 | m4, is4 = m4;  // bit j: the piece at xb + j is listed; it has four bytes
    const uint32_t n_mid = (uint32_t)__popc(mid);
    const uint32_t n_sh = (uint32_t)__popc(lst) | (n_mid << 16);
    // the lists: pieces of 3-4 bytes from the front, mid pieces from the
    // back, x | (len - 1) << 12, in text order (a block scan of the
    // per-thread counts, both packed in one word)
    uint32_t n_list, n_mids;
    {
      uint32_t a = n_sh;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, a, o);
        if (lane >= o) a += y;
      }
      if (lane == 31) sm.warp_tot[ETHREADS / 32 + warp] = a;
      __syncthreads();
      uint32_t before = 0, all = 0;
#pragma unroll
      for (int w = 0; w < ETHREADS / 32; w++) {
        const uint32_t t = sm.warp_tot[ETHREADS / 32 + w];
        before += w < warp ? t : 0u;
        all += t;
      }
      n_list = all & 0xFFFFu;
      n_mids = all >> 16;
      const uint32_t ex = before + a - n_sh;
      uint32_t q = ex & 0xFFFFu;
      for (uint32_t bits = lst; bits; bits &= bits - 1) {
        const int j = __ffs(bits) - 1;
        sm.list[q++] = (uint16_t)((xb + j) | ((2 + ((is4 >> j) & 1u)) << 12));
      }
      uint32_t qm = ex >> 16;
      uint32_t ml = n_mid ? mlen >> (32 - 4 * n_mid) : 0u;  // the first mid piece's length in the low bits
      for (uint32_t bits = mid; bits; bits &= bits - 1, ml >>= 4) {
        const int j = __ffs(bits) - 1;
        sm.list[LIST_END - 1 - qm++] = (uint16_t)((xb + j) | ((ml & 15u) << 12));
      }
    }
    __syncthreads();
    // 2b. the short pieces, MERGE_U per thread per round with their loads
    //     issued together (every length takes the same code path)
    {
      const MergeTabs MT(c.T);
      for (uint32_t i = tid; i < n_list; i += MERGE_U * ETHREADS) {
        Le4 L[MERGE_U];
        int xs[MERGE_U];
#pragma unroll
        for (int u = 0; u < MERGE_U; u++) {
          const uint32_t k = i + u * ETHREADS;
          const uint32_t e = sm.list[k < n_list ? k : i];
          xs[u] = k < n_list ? (int)(e & 0xFFF) : -1;
          L[u] = le4_load(MT, &sm.text[e & 0xFFF], (int)(e >> 12) + 1);
        }
#pragma unroll
        for (int u = 0; u < MERGE_U; u++)
          if (xs[u] >= 0) sm.cnt[xs[u]] = (uint8_t)le4_finish(MT, L[u], &sm.stage[xs[u]]);
      }
      // 2c. mid pieces, one per thread, the parts loop in registers at the
      //     width of the warp's longest piece
      if constexpr (MIDS)
      for (uint32_t b0 = warp * 32; b0 < n_mids; b0 += ETHREADS) {
        const uint32_t i = b0 + lane;
        const bool valid = i < n_mids;
        const uint32_t e = valid ? sm.list[LIST_END - 1 - i] : 0u;
        const int len = valid ? (int)(e >> 12) + 1 : 0;
        const int wmax = __reduce_max_sync(0xffffffffu, len);
        if (!valid) continue;
        const int x = (int)(e & 0xFFF);
        int m;
        if (wmax <= 8) m = merge_reg<8>(MT, &sm.text[x], len, &sm.stage[x]);
        else if (wmax <= 12) m = merge_reg<12>(MT, &sm.text[x], len, &sm.stage[x]);
        else m = merge_reg<16>(MT, &sm.text[x], len, &sm.stage[x]);
        sm.cnt[x] = (uint8_t)m;
      }
    }
    __syncthreads();
    uint32_t my_short = inl;
    const uint32_t my_g = lng;
    for (uint32_t bits = lst | mid; bits; bits &= bits - 1) my_short += sm.cnt[xb + __ffs(bits) - 1];
    {
      const uint32_t ns = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(my));
      if (lane == 0) atomicAdd(&sm.n_starts, ns);
    }
    __syncthreads();
    if (tid == 0) atomicAdd((unsigned long long*)&c.W.status->n_ptok, (unsigned long long)sm.n_starts);
    // 4. per-thread counts (short ids | table entries << 16; a tile has fewer
    //    than 2^16 of each) -> block scan (k_long_fixup adds the table's ids)
    uint32_t th_short = 0, th_g = 0;
    const uint32_t mine = my_short | ((uint32_t)__popc(my_g) << 16);
    {
      uint32_t a = mine;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t ya = __shfl_up_sync(0xffffffffu, a, o);
        if (lane >= o) a += ya;
      }
      if (lane == 31) sm.warp_tot[warp] = a;
      __syncthreads();
      if (tid == 0) {
        uint32_t ra = 0;
        for (int w = 0; w < ETHREADS / 32; w++) {
          const uint32_t ta = sm.warp_tot[w];
          sm.warp_tot[w] = ra;
          ra += ta;
        }
        sm.tile_short = ra;
      }
      __syncthreads();
      const uint32_t ex = sm.warp_tot[warp] + a - mine;
      th_short = ex & 0xFFFFu;
      th_g = ex >> 16;
      sm.th_full[tid] = th_short;
      sm.th_gp[tid] = (uint16_t)th_g;
    }
    __syncthreads();
    const uint32_t tile_short = sm.tile_short & 0xFFFFu, ngp = sm.tile_short >> 16;
    // 5. compaction of short ids (in order, in shared memory); the table
    //    entries (short ids before the piece, its start in the tile) in order
    uint32_t* slot = c.W.staging + tile * STG;
    {
      uint32_t s = th_short, g = th_g;
      for (uint32_t bits = my; bits; bits &= bits - 1) {
        const int x = xb + __ffs(bits) - 1;
        if ((my_g >> (x - xb)) & 1u) {
          *reinterpret_cast<uint4*>(slot + STG - 4 * (g + 1)) = make_uint4(s, (uint32_t)x, 0u, 0u);
          g++;
          continue;
        }
        const uint32_t m = sm.cnt[x];
        for (uint32_t j = 0; j < m; j++) sm.outs[s + j] = sm.stage[x + j];
        s += m;
      }
    }
    __syncthreads();
    // 6. the short ids to the staging slot (16-byte stores: the slot has room
    //    for the rounding before its table); the tile's id count; segment
    //    offsets relative to the tile
    for (uint32_t v = tid; 4 * v < tile_short; v += ETHREADS)
      reinterpret_cast<uint4*>(slot)[v] = reinterpret_cast<const uint4*>(sm.outs)[v];
    if (tid == 0) {
      c.W.tile_count[tile] = tile_short;
      c.W.tile_meta[tile] = tile_short | (ngp << 16);
    }
    for (int64_t s = sm.seg[0] + tid; s < sm.seg[1]; s += ETHREADS) {
      const int64_t x = c.seg_off[s] - t0;
      c.W.seg_rel[s] = (x >= TILE) ? sm.tile_short : ids_before(sm, (int)x);
    }
    __syncthreads();
  }
}

// Adds the table's pieces to the tile counts once their merges are done: per
// tile with table entries (one warp), each entry (in text order) gets its
// source in the arena, its id count and the ids of the tile before it
// (full_excl = short ids before it + the table's ids before it: a warp scan
// over the entries); the tile count grows by the table's ids, and each
// segment offset in the tile by the ids of the entries before it.
constexpr int FIX_BATCH = 4;
__global__ void __launch_bounds__(ETHREADS) k_long_fixup(Call c) {
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t tile = gw; tile < ntiles; tile += nw) {
    const int ngp = (int)(c.W.tile_meta[tile] >> 16);
    if (ngp == 0) continue;
    const int64_t t0 = tile * TILE;
    uint32_t* slot = c.W.staging + tile * STG;
    uint32_t carry = 0;  // the table's ids before this group of entries
    // FIX_BATCH entries per lane per pass, their loads issued together (the
    // entry, then its source, then the count)
    for (int g0 = 0; g0 < ngp; g0 += 32 * FIX_BATCH) {
      uint4 e[FIX_BATCH];
#pragma unroll
      for (int u = 0; u < FIX_BATCH; u++) {
        const int g = g0 + 32 * u + lane;
        e[u] = g < ngp ? *reinterpret_cast<const uint4*>(slot + STG - 4 * (g + 1)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < FIX_BATCH; u++) {
        const int g = g0 + 32 * u + lane;
        if (g < ngp) e[u].z = c.W.gsrc[c.gb + t0 + e[u].y] & ~GSRC_CACHED;
      }
#pragma unroll
      for (int u = 0; u < FIX_BATCH; u++) {
        const int g = g0 + 32 * u + lane;
        e[u].w = g < ngp ? c.W.cnt[e[u].z] : 0u;
      }
#pragma unroll
      for (int u = 0; u < FIX_BATCH; u++) {
        const int g = g0 + 32 * u + lane;
        uint32_t incl = e[u].w;
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (g < ngp) {
          e[u].y = e[u].x + carry + incl - e[u].w;
          *reinterpret_cast<uint4*>(slot + STG - 4 * (g + 1)) = e[u];
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncwarp();
    // segment offsets: short ids | entries before << 16 -> ids before
    const int64_t sg0 = c.W.tile_segs[4 * tile + 1];
    const int64_t sg1 = (tile == ntiles - 1) ? c.S + 1 : c.W.tile_segs[4 * tile + 2];
    for (int64_t sg = sg0 + lane; sg < sg1; sg += 32) {
      const uint32_t v = c.W.seg_rel[sg];
      const uint32_t j = v >> 16;
      uint32_t add = 0;
      if (j > 0) {
        const uint4 e = *reinterpret_cast<const uint4*>(slot + STG - 4 * j);  // entry j - 1
        add = e.y + e.w - e.x;
      }
      c.W.seg_rel[sg] = (v & 0xFFFFu) + add;
    }
    if (lane == 0) c.W.tile_count[tile] += carry;
  }
}

// Ordered output: each tile's staged ids go to out[tile_base + ...], with the
// ids of its table's pieces inserted from the arena.  A tile without table
// entries is one straight copy, COPY_UNROLL ids per thread in flight.  With
// entries the output is a sequence of parts (the short ids before entry 0,
// entry 0's ids, the short ids after it, ...): a shared table holds each
// part's first output and the address of its ids minus that start, a second
// one the part at every 32nd output (one binary search each), so an output
// finds its part in a step or two and reads its id from the staging slot or
// the arena.  Only a tile's last piece can reach past the tile, so a tile
// holds at most one piece of more than HUGE_IDS ids: it is listed for
// k_copy_huge, which spreads it over the grid, and takes no width here (the
// outputs after it shift by its count).  Small CTAs keep many tiles in flight.
constexpr uint32_t HUGE_IDS = 8192;
constexpr int COPY_THREADS = 128;
constexpr int COPY_UNROLL = 24;
// output blocks of 32 ids per tile without its huge piece: the pieces
// inside the tile (at most TILE + 4 ids) and a last one of up to HUGE_IDS
constexpr int COPY_BLK = (TILE + 4 + (int)HUGE_IDS + 31) / 32 + 1;
static_assert((STG * sizeof(uint32_t)) % 16 == 0, "staging slots stay 16-byte aligned");

__global__ void __launch_bounds__(COPY_THREADS, 10) k_copy_out(Call c, int32_t* out, int64_t cap) {
  __shared__ uint32_t s_ps[2 * MAX_GP + 1];           // part starts in the tile's output
  __shared__ unsigned long long s_pp[2 * MAX_GP + 1];  // part address - 4 * start
  __shared__ uint16_t s_blk[COPY_BLK];                 // the part holding output 32 b
  __shared__ uint32_t s_h[2];                          // the huge piece's start and count
  static_assert(2 * MAX_GP + 1 <= 2048, "the block search steps from 1024");
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const int tid = threadIdx.x;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint32_t* slot = c.W.staging + tile * STG;
    const uint64_t base = c.W.tile_base[tile];
    const uint32_t n_out = c.W.tile_base[tile + 1] - (uint32_t)base;
    const uint32_t meta = c.W.tile_meta[tile];
    const int ngp = (int)(meta >> 16);
    if (ngp == 0) {
      for (uint32_t q0 = 0; q0 < n_out; q0 += COPY_UNROLL * COPY_THREADS) {
        uint32_t v[COPY_UNROLL];
#pragma unroll
        for (int k = 0; k < COPY_UNROLL; k++) {
          const uint32_t q = q0 + k * COPY_THREADS + tid;
          v[k] = q < n_out ? __ldcs(slot + q) : 0u;
        }
#pragma unroll
        for (int k = 0; k < COPY_UNROLL; k++) {
          const uint32_t q = q0 + k * COPY_THREADS + tid;
          if (q < n_out && base + q < (uint64_t)cap) out[base + q] = (int32_t)v[k];
        }
      }
      continue;
    }
    // parts: 0 = the short ids before entry 0; 2g + 1 = entry g; 2g + 2 =
    // the short ids after entry g
    const int np = 2 * ngp + 1;
    for (int g = tid; g < ngp; g += COPY_THREADS) {
      const uint4 e = *reinterpret_cast<const uint4*>(slot + STG - 4 * (g + 1));
      const bool huge = e.w > HUGE_IDS;
      const uint32_t rs = huge ? e.y : e.y + e.w;  // where the short ids after it start
      s_ps[2 * g + 1] = e.y;
      s_pp[2 * g + 1] = (unsigned long long)(uintptr_t)(c.W.arena + e.z) - 4ull * e.y;
      s_ps[2 * g + 2] = rs;
      s_pp[2 * g + 2] = (unsigned long long)(uintptr_t)(slot + e.x) - 4ull * rs;
      if (g == ngp - 1) {
        s_h[0] = e.y;
        s_h[1] = huge ? e.w : 0u;
        if (huge) {
          const uint32_t k = atomicAdd(&c.W.status->n_huge, 1u);
          c.W.huge_list[3 * (uint64_t)k] = base + e.y;
          c.W.huge_list[3 * (uint64_t)k + 1] = e.z;
          c.W.huge_list[3 * (uint64_t)k + 2] = e.w;
        }
      }
    }
    if (tid == 0) {
      s_ps[0] = 0;
      s_pp[0] = (unsigned long long)(uintptr_t)slot;
    }
    __syncthreads();
    const uint32_t hst = s_h[0], hcnt = s_h[1];
    const uint32_t n_cmp = n_out - hcnt;  // outputs copied here
    const uint32_t nblk = (n_cmp + 31) >> 5;
    for (uint32_t b = tid; b < nblk; b += COPY_THREADS) {
      int j = 0;  // parts that start at or before output 32 b (part 0 starts at 0)
#pragma unroll
      for (int step = 1024; step > 0; step >>= 1)
        if (j + step <= np && s_ps[j + step - 1] <= 32 * b) j += step;
      s_blk[b] = (uint16_t)(j - 1);
    }
    __syncthreads();
    const bool fits = base + n_out <= (uint64_t)cap;
    for (uint32_t o0 = 0; o0 < n_cmp; o0 += COPY_UNROLL * COPY_THREADS) {
      int32_t v[COPY_UNROLL];
#pragma unroll
      for (int k = 0; k < COPY_UNROLL; k++) {
        const uint32_t o = o0 + k * COPY_THREADS + tid;
        v[k] = 0;
        if (o < n_cmp) {
          int p = s_blk[o >> 5];
          while (p + 1 < np && s_ps[p + 1] <= o) p++;
          v[k] = *reinterpret_cast<const int32_t*>((uintptr_t)(s_pp[p] + 4ull * o));
        }
      }
#pragma unroll
      for (int k = 0; k < COPY_UNROLL; k++) {
        const uint32_t o = o0 + k * COPY_THREADS + tid;
        const uint64_t pos = base + o + (o >= hst ? hcnt : 0u);
        if (o < n_cmp && (fits || pos < (uint64_t)cap)) out[pos] = v[k];
      }
    }
    __syncthreads();
  }
}

// The listed long pieces, each copied by every thread of the grid.
__global__ void __launch_bounds__(ETHREADS) k_copy_huge(Call c, int32_t* out, int64_t cap) {
  const uint32_t n_huge = c.W.status->n_huge;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  const uint64_t me = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (uint32_t k = 0; k < n_huge; k++) {
    const uint64_t o = c.W.huge_list[3 * (uint64_t)k];
    const int32_t* src = c.W.arena + c.W.huge_list[3 * (uint64_t)k + 1];
    const uint64_t cnt = c.W.huge_list[3 * (uint64_t)k + 2];
    for (uint64_t j0 = 0; j0 < cnt; j0 += 4 * stride) {
      int32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const uint64_t j = j0 + u * stride + me;
        v[u] = j < cnt ? __ldcs(src + j) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const uint64_t j = j0 + u * stride + me;
        if (j < cnt && o + j < (uint64_t)cap) out[o + j] = v[u];
      }
    }
  }
}

// out_offsets[s] = the tile base of the tile that holds segment s's start plus
// the ids before it in that tile; n_ids = total.
// With id_base (a batch of a pipelined call) every offset is shifted by
// *id_base, and id_base[1] = *id_base + n_ids.
__global__ void k_seg_offsets(Call c, int64_t* out_offsets, int64_t* id_base) {
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const int64_t b = id_base ? id_base[0] : 0;
  for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s <= c.S;
       s += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = min(c.seg_off[s] / TILE, ntiles - 1);
    out_offsets[s] = b + (int64_t)c.W.tile_base[tile] + c.W.seg_rel[s];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    c.W.status->n_ids = c.W.tile_base[ntiles];
    c.W.status->n_long = c.W.status->n_medium + c.W.status->n_biglong + c.W.status->n_cl;
    if (id_base) id_base[1] = b + c.W.tile_base[ntiles];
  }
}

// off[i] = raw[i] - raw[0]: a batch's segment offsets made relative to its text.
__global__ void k_rebase(const int64_t* raw, int64_t* off, int64_t cnt) {
  const int64_t r0 = raw[0];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < cnt; i += (int64_t)gridDim.x * blockDim.x)
    off[i] = raw[i] - r0;
}

// End of the pre-token that starts at byte p: the next start bit, else the
// first start of a later split tile, else n (reads the start bitmap).
__device__ int64_t piece_end(const Call& c, int64_t p, int64_t ntiles) {
  constexpr int B = 8;  // bitmap words (or tile firsts) loaded together per step
  const int64_t tile = p / TILE;
  const int64_t tend = min(c.n, (tile + 1) * TILE);
  int64_t y = p + 1;
  if (y < tend) {
    const uint32_t w = c.W.pbits[y >> 5] >> (y & 31);
    if (w) return min(c.n, y + __ffs(w) - 1);
    const int64_t wend = (tend + 31) >> 5;  // the tile's words (tiles are whole words)
    for (int64_t wi = (y >> 5) + 1; wi < wend; wi += B) {
      uint32_t v[B];
#pragma unroll
      for (int k = 0; k < B; k++) v[k] = wi + k < wend ? c.W.pbits[wi + k] : 0u;
#pragma unroll
      for (int k = 0; k < B; k++)
        if (v[k]) return min(c.n, ((wi + k) << 5) + __ffs(v[k]) - 1);
    }
  }
  for (int64_t k0 = tile + 1; k0 < ntiles; k0 += B) {
    uint32_t f[B];
#pragma unroll
    for (int k = 0; k < B; k++) f[k] = k0 + k < ntiles ? c.W.tile_first[k0 + k] : NO_START;
#pragma unroll
    for (int k = 0; k < B; k++)
      if (f[k] != NO_START) return (k0 + k) * TILE + f[k];
  }
  return c.n;
}

// Pre-tokens longer than SHORT_MAX bytes -> three work lists (medium: one warp
// each, big: one CTA each, longest: one CTA cluster each), as (start, length)
// pairs.
__device__ __forceinline__ void list_long(const Call& c, int64_t p, int64_t len) {
  if (len <= MEDIUM_MAX) {
    const uint32_t k = atomicAdd(&c.W.status->n_medium, 1u);
    c.W.long_list[2 * k] = (uint32_t)p;
    c.W.long_list[2 * k + 1] = (uint32_t)len;
  } else if (len <= CLUSTER_MIN) {
    const uint32_t k = atomicAdd(&c.W.status->n_biglong, 1u);
    c.W.big_list[2 * k] = (uint32_t)p;
    c.W.big_list[2 * k + 1] = (uint32_t)len;
  } else {
    const uint32_t k = atomicAdd(&c.W.status->n_cl, 1u);
    c.W.cl_list[2 * k] = (uint32_t)p;
    c.W.cl_list[2 * k + 1] = (uint32_t)len;
  }
}

// The pre-tokens of MID_MIN bytes or more: mid pieces (up to SHORT_MAX
// bytes) -> mid_list when they are merged on the side streams (mid_side; up
// to 8 bytes from the front and longer ones from the back: k_merge_mid gives
// a warp one of the two), else the tile kernel merges them; longer ones ->
// list_long.
// Each thread reads FIND_WPT words of the start bitmap; a start's length is
// the distance to the next start bit (the next word is in reach of every
// start of the word; the text end counts as a start), else piece_end.  The
// mid entries of a warp take one atomic per list: a count pass, a warp scan,
// then a write pass.  Specials are one id each, left to the tile kernel.
constexpr int FIND_WPT = 4;
__global__ void __launch_bounds__(256) k_find_long(Call c) {
  const int lane = threadIdx.x & 31;
  const int64_t ntiles = (c.n + TILE - 1) / TILE;
  const int64_t nwords = (c.n + 31) >> 5;
  const int64_t nch = (nwords + FIND_WPT - 1) / FIND_WPT;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b0 = blockIdx.x * (int64_t)blockDim.x + (threadIdx.x & ~31); b0 < nch; b0 += stride) {
    const int64_t ch = b0 + lane;
    uint32_t ia = 0, ib = 0;
    for (int pass = 0; pass < 2; pass++) {
      if (pass == 1) {
        // exclusive warp scans of the counts, one atomic per list
        uint32_t sa = ia, sb = ib;
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t ya = __shfl_up_sync(0xffffffffu, sa, o), yb = __shfl_up_sync(0xffffffffu, sb, o);
          if (lane >= o) { sa += ya; sb += yb; }
        }
        uint32_t ba = 0, bb = 0;
        if (lane == 31) {
          if (sa) ba = atomicAdd(&c.W.status->n_mid_a, sa);
          if (sb) bb = atomicAdd(&c.W.status->n_mid_b, sb);
        }
        ba = __shfl_sync(0xffffffffu, ba, 31);
        bb = __shfl_sync(0xffffffffu, bb, 31);
        ia = ba + sa - ia;
        ib = bb + sb - ib;
      }
      // the thread's words, the one after them and their special starts,
      // loaded together
      uint32_t pw[FIND_WPT + 1], sw[FIND_WPT];
#pragma unroll
      for (int k = 0; k <= FIND_WPT; k++) {
        const int64_t wi = ch * FIND_WPT + k;
        pw[k] = (ch < nch && wi < nwords) ? c.W.pbits[wi] : 0u;
        if (k < FIND_WPT) sw[k] = (c.T.n_spec && ch < nch && wi < nwords) ? c.W.sbits[wi] : 0u;
      }
#pragma unroll
      for (int k = 0; k < FIND_WPT; k++) {
        const int64_t wi = ch * FIND_WPT + k;
        if (ch >= nch || wi >= nwords) break;
        uint32_t bits = pw[k];
        if ((wi << 5) + 32 > c.n) bits &= (1u << (c.n - (wi << 5))) - 1u;
        if (!bits) continue;
        uint64_t w = bits;
        if ((wi << 5) + 32 < c.n) {
          uint32_t nx = pw[k + 1];
          if ((wi << 5) + 64 > c.n) nx |= ~((1u << (c.n - (wi << 5) - 32)) - 1u);
          w |= (uint64_t)nx << 32;
        } else {
          w |= ~0ull << (c.n - (wi << 5));
        }
        static_assert(MID_MIN == 5 && SHORT_MAX <= 32, "one look at the next word covers SHORT_MAX");
        const uint64_t near4 = (w >> 1) | (w >> 2) | (w >> 3) | (w >> 4);
        for (uint32_t cand = bits & ~(uint32_t)near4 & ~sw[k]; cand; cand &= cand - 1) {
          const int x = __ffs(cand) - 1;
          const int64_t p = (wi << 5) + x;
          const uint64_t nxt = w >> (x + 1);
          const int d = nxt ? __ffsll((long long)nxt) : 0;  // length, if the next start is in w
          if (d >= MID_MIN && d <= SHORT_MAX) {
            if (!c.W.mid_side) continue;
            if (pass == 0) {
              if (d <= 8) ia++;
              else ib++;
            } else if (d <= 8) {
              c.W.mid_list[2 * (int64_t)ia] = (uint32_t)p;
              c.W.mid_list[2 * (int64_t)ia + 1] = (uint32_t)d;
              ia++;
            } else {
              const int64_t e = c.W.mid_cap - 1 - ib;
              c.W.mid_list[2 * e] = (uint32_t)p;
              c.W.mid_list[2 * e + 1] = (uint32_t)d;
              ib++;
            }
          } else if (pass == 1) {
            const int64_t len = d ? d : piece_end(c, p, ntiles) - p;
            if (len > SHORT_MAX) list_long(c, p, len);
          }
        }
      }
    }
  }
}

// Word cache of the long pieces ("tokenizers v1 ...", "Key Technical
// Improvements": a repeated word is merged only once).  One warp per listed
// piece hashes its bytes, then claims a slot of the table or finds the slot
// of an identical piece (same length, bytes compared one by one), so each
// distinct long piece is merged once and its copies point at it.
__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 33;
  x *= 0xff51afd7ed558ccdull;
  x ^= x >> 33;
  x *= 0xc4ceb9fe1a85ec53ull;
  x ^= x >> 33;
  return x;
}

// Order-free hash of the bytes text[p .. p+len): a sum over 8-byte groups,
// each mixed with its position, so any split of the groups among threads
// gives the same value.  Returns this thread's partial sum over groups
// first, first + step, ...
__device__ __forceinline__ uint64_t hash_part(const Call& c, int64_t p, int64_t len, int64_t first,
                                              int64_t step) {
  uint64_t h = 0;
  for (int64_t g = first; 8 * g < len; g += step) {
    const int64_t q = 8 * g;
    uint64_t v = 0;
    for (int j = 0; j < 8 && q + j < len; j++) v |= (uint64_t)gbyte(c, p + q + j) << (8 * j);
    h += mix64(v ^ (0x9E3779B97F4A7C15ull * (uint64_t)(q + 1)));
  }
  return h;
}

// Claims a slot for (key, p, len) or finds the slot of an identical piece.
// Run by all lanes of a warp (medium pieces) or all threads of a CTA (big);
// `eq` compares the bytes with a candidate owner across the group.  Returns
// the start of the piece whose merge p uses.
template <class Eq>
__device__ int64_t dedup_claim(const Call& c, uint64_t key, int64_t p, int64_t len, bool leader,
                               uint64_t* shared_word, Eq eq, bool cta) {
  const uint64_t mask = (1ull << c.W.dtab_log2) - 1;
  uint64_t slot = key & mask;
  for (int probe = 0; probe < 64; probe++, slot = (slot + 1) & mask) {
    // one thread claims or reads the slot, then the owner word; all share it
    if (leader) {
      const unsigned long long old = atomicCAS(&c.W.dtab[2 * slot], 0ull, (unsigned long long)key);
      uint64_t r;
      if (old == 0) {
        st_release_u64(reinterpret_cast<uint64_t*>(&c.W.dtab[2 * slot + 1]),
                       (uint64_t)(c.gb + p + 1) | ((uint64_t)len << 32));
        r = 1;  // claimed
      } else if (old != key) {
        r = 2;  // another key: next slot
      } else {
        uint64_t ow = 0;
        for (uint32_t spins = 0; spins < SPIN_LIMIT; spins++) {
          ow = ld_acquire_u64(reinterpret_cast<const uint64_t*>(&c.W.dtab[2 * slot + 1]));
          if (ow) break;
          __nanosleep(32);
        }
        r = ow ? ow : 3;  // 3: gave up waiting
      }
      *shared_word = r;
    }
    if (cta) __syncthreads();
    else __syncwarp();
    const uint64_t r = *shared_word;
    if (cta) __syncthreads();
    else __syncwarp();
    if (r == 1 || r == 3) return c.gb + p;  // owner (or give up: merge this copy itself)
    if (r == 2) continue;
    const int64_t owner = (int64_t)(r & 0xFFFFFFFFu) - 1;
    if ((int64_t)(r >> 32) != len) continue;
    if (eq(owner)) return owner;
  }
  return c.gb + p;
}

__global__ void k_dedup_medium(Call c) {
  __shared__ uint64_t s_word[ETHREADS / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t n_med = c.W.status->n_medium;
  for (int64_t k = gw; k < n_med; k += nw) {
    const int64_t p = c.W.long_list[2 * k], len = c.W.long_list[2 * k + 1];
    uint64_t h = hash_part(c, p, len, lane, 32);
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    const uint64_t key = mix64(h ^ (uint64_t)len) | 1ull;
    auto eq = [&](int64_t owner) {
      bool same = true;
      for (int64_t q = lane; q < len && same; q += 32) same = gbyte(c, p + q) == text_at(c, owner + q);
      return (bool)__all_sync(0xffffffffu, same);
    };
    const int64_t src = dedup_claim(c, key, p, len, lane == 0, &s_word[warp], eq, false);
    if (lane == 0) {
      c.W.gsrc[c.gb + p] = (uint32_t)src;
      c.W.long_key[k] = key;
    }
  }
}

__global__ void __launch_bounds__(1024) k_dedup_big(Call c) {
  __shared__ uint64_t s_red[32];
  __shared__ uint64_t s_word;
  __shared__ uint32_t s_idx;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t n_big = c.W.status->n_biglong, n_cl = c.W.status->n_cl;
  for (;;) {
    if (tid == 0) s_idx = atomicAdd(&c.W.status->dedup_big_next, 1u);
    __syncthreads();
    const uint32_t k = s_idx;
    __syncthreads();
    if (k >= n_big + n_cl) break;
    const uint32_t* ent = k < n_big ? &c.W.big_list[2 * k] : &c.W.cl_list[2 * (k - n_big)];
    const int64_t p = ent[0], len = ent[1];
    uint64_t h = hash_part(c, p, len, tid, blockDim.x);
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if (lane == 0) s_red[warp] = h;
    __syncthreads();
    h = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) h += s_red[w];
    __syncthreads();
    const uint64_t key = mix64(h ^ (uint64_t)len) | 1ull;
    auto eq = [&](int64_t owner) {
      bool same = true;
      for (int64_t q = tid; q < len && same; q += blockDim.x) same = gbyte(c, p + q) == text_at(c, owner + q);
      return (bool)__syncthreads_and(same);
    };
    const int64_t src = dedup_claim(c, key, p, len, tid == 0, &s_word, eq, true);
    if (tid == 0) {
      c.W.gsrc[c.gb + p] = (uint32_t)src;
      if (k < n_big) c.W.big_key[k] = key;
      else c.W.cl_key[k - n_big] = key;
    }
  }
}

// --------------------------------------------------------------------------
// Cross-call word cache.  k_cache_lookup: every distinct listed piece of
// this call (an owner) whose key, length and bytes match a cache entry takes
// the entry's ids (gsrc gets GSRC_CACHED, so the merge kernels pass it by).
// k_cache_insert: every owner merged in this call enters the cache while
// its capacity lasts.  One warp per listed piece.
__device__ __forceinline__ bool listed_piece(const Call& c, uint64_t k, int64_t* p, int64_t* len, uint64_t* key) {
  const uint64_t n_med = c.W.status->n_medium, n_big = c.W.status->n_biglong, n_cl = c.W.status->n_cl;
  if (k < n_med) {
    *p = c.W.long_list[2 * k]; *len = c.W.long_list[2 * k + 1]; *key = c.W.long_key[k];
  } else if (k < n_med + n_big) {
    k -= n_med;
    *p = c.W.big_list[2 * k]; *len = c.W.big_list[2 * k + 1]; *key = c.W.big_key[k];
  } else if (k < n_med + n_big + n_cl) {
    k -= n_med + n_big;
    *p = c.W.cl_list[2 * k]; *len = c.W.cl_list[2 * k + 1]; *key = c.W.cl_key[k];
  } else {
    return false;
  }
  return true;
}

// Group-wide compare of a piece's bytes with a cache entry and copy of its
// ids (a warp for pieces of up to MEDIUM_MAX bytes, a CTA beyond): no early
// exit, so the loads of many positions are in flight at once.
template <bool CTA>
__device__ void cache_probe(const Call& c, int64_t G, int64_t len, uint64_t key, uint64_t* s_ref) {
  const CacheDev& C = c.W.cache;
  const uint64_t mask = (1ull << C.slot_log2) - 1;
  const int t = CTA ? (int)threadIdx.x : (int)(threadIdx.x & 31);
  const int nt = CTA ? (int)blockDim.x : 32;
  uint64_t slot = key & mask;
  for (int probe = 0; probe < 64; probe++, slot = (slot + 1) & mask) {
    // one thread reads the slot; all share (entry + 1, or 0 to stop, or ~0 to go on)
    if (t == 0) {
      const uint64_t sk = C.slots[2 * slot];
      uint64_t r = 0;
      if (sk != 0) {
        r = ~0ull;
        const uint64_t ref = sk == key ? C.slots[2 * slot + 1] : 0;
        if (ref && (int64_t)C.entries[ref - 1].len == len) r = ref;
      }
      *s_ref = r;
    }
    if (CTA) __syncthreads();
    else __syncwarp();
    const uint64_t ref = *s_ref;
    if (CTA) __syncthreads();
    else __syncwarp();
    if (ref == 0) return;  // not cached
    if (ref == ~0ull) continue;
    const CacheEntry e = C.entries[ref - 1];
    bool same = true;
    for (int64_t q = t; q < len; q += nt) same &= C.bytes[e.byte_off + q] == text_at(c, G + q);
    const bool all = CTA ? __syncthreads_and(same) : __all_sync(0xffffffffu, same);
    if (!all) continue;
    for (uint32_t j = t; j < e.n_ids; j += nt) c.W.arena[G + j] = C.ids[e.id_off + j];
    if (t == 0) {
      c.W.cnt[G] = e.n_ids;
      c.W.gsrc[G] = (uint32_t)G | GSRC_CACHED;
      atomicAdd(&c.W.status->n_cache_hits, 1u);
    }
    return;
  }
}

// Pieces of up to MEDIUM_MAX bytes: one warp each.
__global__ void k_cache_lookup(Call c) {
  __shared__ uint64_t s_ref[ETHREADS / 32];
  const uint64_t gw = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint64_t n_med = c.W.status->n_medium;
  for (uint64_t k = gw; k < n_med; k += nw) {
    const int64_t p = c.W.long_list[2 * k], len = c.W.long_list[2 * k + 1];
    const int64_t G = c.gb + p;
    if (c.W.gsrc[G] != (uint32_t)G) continue;  // a copy of another piece of this call
    cache_probe<false>(c, G, len, c.W.long_key[k], &s_ref[threadIdx.x >> 5]);
  }
}

// Longer pieces: one CTA each.
__global__ void __launch_bounds__(1024) k_cache_lookup_big(Call c) {
  __shared__ uint64_t s_ref;
  const uint64_t n_big = c.W.status->n_biglong, n_cl = c.W.status->n_cl;
  for (uint64_t k = blockIdx.x; k < n_big + n_cl; k += gridDim.x) {
    const uint32_t* ent = k < n_big ? &c.W.big_list[2 * k] : &c.W.cl_list[2 * (k - n_big)];
    const uint64_t key = k < n_big ? c.W.big_key[k] : c.W.cl_key[k - n_big];
    const int64_t G = c.gb + ent[0], len = ent[1];
    if (c.W.gsrc[G] != (uint32_t)G) continue;
    cache_probe<true>(c, G, len, key, &s_ref);
  }
}

__global__ void k_cache_insert(Call c) {
  const int lane = threadIdx.x & 31;
  const uint64_t gw = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const CacheDev& C = c.W.cache;
  const uint64_t mask = (1ull << C.slot_log2) - 1;
  int64_t p, len;
  uint64_t key;
  for (uint64_t k = gw; listed_piece(c, k, &p, &len, &key); k += nw) {
    const int64_t G = c.gb + p;
    if (c.W.gsrc[G] != (uint32_t)G) continue;  // a copy, or taken from the cache
    const uint32_t n_ids = c.W.cnt[G];
    // reserve an entry, the bytes and the ids (a failed reservation is not
    // returned: the cache counts as full from then on)
    unsigned long long e = 0, bo = 0, io = 0;
    if (lane == 0) {
      e = atomicAdd(&C.used[0], 1ull);
      bo = atomicAdd(&C.used[1], (unsigned long long)len);
      io = atomicAdd(&C.used[2], (unsigned long long)n_ids);
    }
    e = __shfl_sync(0xffffffffu, e, 0);
    bo = __shfl_sync(0xffffffffu, bo, 0);
    io = __shfl_sync(0xffffffffu, io, 0);
    if (e >= C.max_entries || bo + len > C.max_bytes || io + n_ids > C.max_ids) continue;
    for (int64_t q = lane; q < len; q += 32) C.bytes[bo + q] = text_at(c, G + q);
    for (uint32_t j = lane; j < n_ids; j += 32) C.ids[io + j] = c.W.arena[G + j];
    if (lane == 0) {
      C.entries[e] = CacheEntry{bo, io, (uint32_t)len, n_ids};
      uint64_t slot = key & mask;
      for (int probe = 0; probe < 64; probe++, slot = (slot + 1) & mask) {
        if (atomicCAS(&C.slots[2 * slot], 0ull, (unsigned long long)key) == 0ull) {
          C.slots[2 * slot + 1] = e + 1;  // read by later calls only (stream order)
          atomicAdd(&c.W.status->n_cache_inserts, 1u);
          break;
        }
      }
    }
  }
}

// The parts loop of one pre-token of SMALL_WARP_MAX bytes or fewer on one
// warp, in registers: element i sits in lane i % 32, slot i / 32 (K slots).
// Each step takes the leftmost pair of least rank by a warp reduction of
// (rank << 6 | position), merges it, shifts the later elements down one
// place, and looks up the two new neighbour pairs in two lanes at once.
// ids -> dst[0 ..]; returns the count.
constexpr int SMALL_WARP_MAX = 128;
// the value of slot s (uniform across the warp) of a per-lane array
template <int K>
__device__ __forceinline__ uint32_t slot_of(const uint32_t (&v)[K], int s) {
  uint32_t r = v[0];
#pragma unroll
  for (int k = 1; k < K; k++) r = s == k ? v[k] : r;
  return r;
}
template <int K>
__device__ int merge_warp(const Call& c, int64_t s, int n, uint32_t* dst) {
  static_assert(K >= 1 && K <= 4, "one to four elements per lane (positions in seven bits)");
  const int lane = threadIdx.x & 31;
  constexpr uint32_t NOKEY = 0xFFFFFFFFu;
  uint32_t id[K], rk[K];
#pragma unroll
  for (int k = 0; k < K; k++) {
    const int i = 32 * k + lane;
    const uint32_t b = gbyte(c, s + i);
    id[k] = i < n ? __ldg(&c.T.byte_id[b]) : 0u;
    rk[k] = (i + 1 < n) ? __ldg(&c.T.dense[(b << 8) | gbyte(c, s + i + 1)]) : RANK_MAX;
  }
  int m = n;
  for (int step = 0; step < n; step++) {
    uint32_t key = NOKEY;
#pragma unroll
    for (int k = 0; k < K; k++) {
      const int i = 32 * k + lane;
      if (i + 1 < m && rk[k] != RANK_MAX) key = min(key, (rk[k] << 7) | (uint32_t)i);
    }
    for (int o = 16; o > 0; o >>= 1) key = min(key, __shfl_xor_sync(0xffffffffu, key, o));
    if (key == NOKEY) break;
    const uint32_t rs = key >> 7;
    const int j = (int)(key & 127);
    // element j becomes rs; elements after j move down one place
#pragma unroll
    for (int k = 0; k < K; k++) {
      const uint32_t nid = __shfl_down_sync(0xffffffffu, id[k], 1);
      const uint32_t nrk = __shfl_down_sync(0xffffffffu, rk[k], 1);
      const uint32_t wid = (k + 1 < K) ? __shfl_sync(0xffffffffu, id[(k + 1) % K], 0) : 0u;
      const uint32_t wrk = (k + 1 < K) ? __shfl_sync(0xffffffffu, rk[(k + 1) % K], 0) : RANK_MAX;
      const int i = 32 * k + lane;
      if (i > j) {
        id[k] = lane == 31 ? wid : nid;
        rk[k] = lane == 31 ? wrk : nrk;
      } else if (i == j) {
        id[k] = rs;
      }
    }
    m--;
    // neighbours of the new element: j - 1 and j + 1 (after the shift)
    const int jl = j - 1, jr = j + 1;
    const uint32_t idl = jl >= 0 ? __shfl_sync(0xffffffffu, slot_of<K>(id, jl >> 5), jl & 31) : 0u;
    const uint32_t idr = jr < m ? __shfl_sync(0xffffffffu, slot_of<K>(id, jr >> 5), jr & 31) : 0u;
    const bool do_l = jl >= 0 && lane == (jl & 31);
    const bool do_r = lane == (j & 31);
    // one call site, so the two lanes' lookups run together (ranks < 2^20)
    uint32_t r = RANK_MAX;
    if (do_l || (do_r && jr < m)) r = pair_rank(c.T, do_l ? idl : rs, do_l ? rs : idr);
#pragma unroll
    for (int k = 0; k < K; k++) {
      if (do_l && 32 * k + lane == jl) rk[k] = r;
      if (do_r && 32 * k + lane == j) rk[k] = r;
    }
  }
#pragma unroll
  for (int k = 0; k < K; k++) {
    const int i = 32 * k + lane;
    if (i < m) dst[i] = id[k];
  }
  return m;
}

// Merges the listed pieces that are the first of their kind (see the word
// cache above).  k_merge_big: one 1024-thread CTA per piece over MEDIUM_MAX
// bytes; k_merge_medium: one warp per piece of SHORT_MAX+1..MEDIUM_MAX bytes
// (in registers up to SMALL_WARP_MAX bytes, else and for runs of one byte the
// round merge).
// ids -> arena[start ..], count -> cnt[start].
constexpr int BIG_THREADS = 1024;
constexpr int64_t BIG_FIRST = 8192;
// Parts a big merge holds in shared memory: its rounds move there once the
// piece has shrunk to this many parts (at once for pieces this short).
constexpr int64_t BIG_SCAP = 25600;
constexpr int BIG_SMEM = (int)(BIG_SCAP * CHUNK_PART);
__global__ void __launch_bounds__(BIG_THREADS) k_merge_big(Call c) {
  __shared__ ChunkSh<BIG_THREADS / 32> s_ch;
  __shared__ uint32_t s_idx;
  extern __shared__ __align__(16) uint8_t s_parts[];
  const int tid = threadIdx.x;
  const uint32_t n_big = c.W.status->n_biglong;
  // two passes over the list, pieces over BIG_FIRST bytes first, so that no
  // CTA starts a long piece late (longest-first scheduling, in two buckets)
  for (int pass = 0; pass < 2; pass++) {
    uint32_t* next = pass == 0 ? &c.W.status->big_next : &c.W.status->big_next2;
    for (;;) {
      if (tid == 0) s_idx = atomicAdd(next, 1u);
      __syncthreads();
      const uint32_t k = s_idx;
      __syncthreads();
      if (k >= n_big) break;
      const int64_t p = c.W.big_list[2 * k], len = c.W.big_list[2 * k + 1];
      if ((len > BIG_FIRST) != (pass == 0)) continue;
      if (c.W.gsrc[c.gb + p] != (uint32_t)(c.gb + p)) continue;  // a copy: uses its owner's ids
      const int64_t m = merge_chunks<BIG_THREADS / 32>(c, p, len, s_parts, BIG_SCAP, s_ch);
      if (tid == 0) c.W.cnt[c.gb + p] = (uint32_t)m;
    }
  }
}

// k_merge_cluster: one cluster of MERGE_CL CL_THREADS-thread CTAs per piece
// over CLUSTER_MIN bytes; rank 0 takes the next piece and shares it through
// distributed shared memory.
constexpr int CL_THREADS = 1024;
__global__ void __cluster_dims__(MERGE_CL, 1, 1) __launch_bounds__(CL_THREADS, 1024 / CL_THREADS) k_merge_cluster(Call c) {
  __shared__ int64_t s64[33];
  __shared__ uint32_t s32[33];
  __shared__ uint32_t s_idx;
  const uint32_t rank = cl_rank();
  const uint32_t n_cl = c.W.status->n_cl;
  for (;;) {
    if (rank == 0 && threadIdx.x == 0) s_idx = atomicAdd(&c.W.status->cl_next, 1u);
    cl_sync();
    const uint32_t k = cl_ld32(cl_map(&s_idx, 0));
    cl_sync();
    if (k >= n_cl) break;
    const int64_t p = c.W.cl_list[2 * k], len = c.W.cl_list[2 * k + 1];
    if (c.W.gsrc[c.gb + p] != (uint32_t)(c.gb + p)) continue;  // a copy: uses its owner's ids
    const int64_t m = merge_rounds(c, CGroup<MERGE_CL, CL_THREADS / 32>{s64, s32, rank}, p, len);
    if (rank == 0 && threadIdx.x == 0) c.W.cnt[c.gb + p] = (uint32_t)m;
  }
}

__global__ void __launch_bounds__(ETHREADS) k_merge_medium(Call c) {
  const int lane = threadIdx.x & 31;
  const uint32_t n_med = c.W.status->n_medium;
  for (;;) {
    uint32_t k = 0;
    if (lane == 0) k = atomicAdd(&c.W.status->medium_next, 1u);
    k = __shfl_sync(0xffffffffu, k, 0);
    if (k >= n_med) break;
    const int64_t p = c.W.long_list[2 * k], len = c.W.long_list[2 * k + 1];
    if (c.W.gsrc[c.gb + p] != (uint32_t)(c.gb + p)) continue;  // a copy: uses its owner's ids
    int64_t m;
    uint32_t* dst = reinterpret_cast<uint32_t*>(c.W.arena + c.gb + p);
    // a run of one repeated byte (white space, "----") merges in a few
    // rounds; other pieces of up to SMALL_WARP_MAX bytes one merge at a time
    bool run = true;
    const uint32_t b0 = gbyte(c, p);
    for (int64_t q = lane; q < len; q += 32) run &= gbyte(c, p + q) == b0;
    run = __all_sync(0xffffffffu, run);
    if (run || len > SMALL_WARP_MAX) m = merge_rounds(c, RGroup<1>{nullptr, nullptr}, p, len);
    else if (len <= 32) m = merge_warp<1>(c, p, (int)len, dst);
    else if (len <= 64) m = merge_warp<2>(c, p, (int)len, dst);
    else if (len <= 96) m = merge_warp<3>(c, p, (int)len, dst);
    else m = merge_warp<4>(c, p, (int)len, dst);
    if (lane == 0) c.W.cnt[c.gb + p] = (uint32_t)m;
  }
}

// Word cache of the mid pieces (MID_MIN..SHORT_MAX bytes): a repeated word
// is merged once.  The key is the piece's bytes themselves (two words,
// zero-padded), so equal keys of equal length are equal pieces and no byte
// comparison is needed.  Slot: key0 + 1 (0 = empty; claimed by CAS), key1,
// then (owner G + 1) | len << 32 published with release.  Each word is
// written once per call (k_clear_mtab clears them in an earlier kernel), so a
// plain load, which may hit a stale L1 line, returns either 0 or the final
// value: frequent words are then found in L1 without an atomic, and only a
// slot that reads empty is claimed by CAS (a hot word's slot would otherwise
// serialise hundreds of thousands of atomics).  Returns the start of the
// piece whose ids p uses (G itself for the first occurrence, or when the
// table is full or a wait gives up).
__device__ int64_t mid_claim(const Call& c, uint64_t k0, uint64_t k1, int len, int64_t G) {
  const uint64_t key = k0 + 1;  // 0 only for 8 bytes of 0xFF: not cached
  if (key == 0) return G;
  const uint64_t mask = (1ull << c.W.mtab_log2) - 1;
  uint64_t slot = mix64(k0 ^ mix64(k1 ^ (uint64_t)len)) & mask;
  for (int probe = 0; probe < 32; probe++, slot = (slot + 1) & mask) {
    unsigned long long* e = c.W.mtab + 4 * slot;
    unsigned long long cur = e[0];
    if (cur == 0) {
      cur = atomicCAS(&e[0], 0ull, (unsigned long long)key);
      if (cur == 0) {
        e[1] = k1;
        st_release_u64(reinterpret_cast<uint64_t*>(&e[2]), (uint64_t)(G + 1) | ((uint64_t)len << 32));
        return G;
      }
    }
    if (cur != key) continue;
    uint64_t v = e[2];
    for (uint32_t spins = 0; v == 0 && spins < SPIN_LIMIT; spins++) {
      v = ld_acquire_u64(reinterpret_cast<const uint64_t*>(&e[2]));
      if (!v) __nanosleep(32);
    }
    if (!v) return G;
    if ((int)(v >> 32) != len) continue;
    const int64_t owner = (int64_t)(v & 0xFFFFFFFFu) - 1;
    if (len <= 8) return owner;  // key0 holds every byte
    // key1: a plain load is 0 or final; 0 (or a mismatch) is confirmed coherently
    uint64_t w1 = e[1];
    if (w1 != k1 || k1 == 0) w1 = ld_acquire_u64(reinterpret_cast<const uint64_t*>(&e[1]));
    if (w1 == k1) return owner;
  }
  return G;
}

// Clears the mid-piece word cache of this call (every word: a waiter must
// never see an owner left by an earlier call).  Runs on the mid-piece stream,
// off the split's critical path.
__global__ void k_clear_mtab(Work W) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (1ll << W.mtab_log2);
       i += (int64_t)gridDim.x * blockDim.x) {
    reinterpret_cast<uint4*>(W.mtab)[2 * i] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(W.mtab)[2 * i + 1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// One thread per listed mid piece: its source (gsrc) from the word cache;
// the first occurrences go to mid_own (front or back like mid_list, one
// atomic per warp).
template <bool BACK>
__global__ void __launch_bounds__(ETHREADS) k_dedup_mid(Call c) {
  const int lane = threadIdx.x & 31;
  const int64_t nm = BACK ? c.W.status->n_mid_b : c.W.status->n_mid_a;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b0 = blockIdx.x * (int64_t)blockDim.x + (threadIdx.x & ~31); b0 < nm; b0 += stride) {
    const int64_t i = b0 + lane;
    bool own = false;
    uint32_t p = 0, len = 0;
    if (i < nm) {
      const int64_t k = BACK ? c.W.mid_cap - 1 - i : i;
      p = c.W.mid_list[2 * k];
      len = c.W.mid_list[2 * k + 1];
      uint64_t k0 = 0, k1 = 0;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        k0 |= (uint64_t)((uint32_t)j < len ? gbyte(c, (int64_t)p + j) : 0) << (8 * j);
        if (BACK) k1 |= (uint64_t)((uint32_t)(j + 8) < len ? gbyte(c, (int64_t)p + j + 8) : 0) << (8 * j);
      }
      const int64_t G = c.gb + p;
      const int64_t src = mid_claim(c, k0, k1, (int)len, G);
      c.W.gsrc[G] = (uint32_t)src;
      own = src == G;
    }
    const uint32_t om = __ballot_sync(0xffffffffu, own);
    uint32_t base = 0;
    if (lane == 0 && om) base = atomicAdd(BACK ? &c.W.status->n_own_b : &c.W.status->n_own_a, (uint32_t)__popc(om));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (own) {
      const int64_t r = base + __popc(om & ((1u << lane) - 1u));
      const int64_t k = BACK ? c.W.mid_cap - 1 - r : r;
      c.W.mid_own[2 * k] = p;
      c.W.mid_own[2 * k + 1] = len;
    }
  }
}

// The distinct mid pieces (every mid piece when the call does not use the
// word cache, each then its own source): one thread each over the whole
// grid, the register loop of the width the warp's longest piece needs (the
// front of the list: up to 8 bytes, BACK = false; its back: 12 or 16), one
// launch each so that the narrow loop runs at its own occupancy.  Ids to the
// arena at the piece's start, the count beside them.
template <bool BACK>
__global__ void __launch_bounds__(ETHREADS) k_merge_mid(Call c) {
  const MergeTabs MT(c.T);
  const int lane = threadIdx.x & 31;
  const bool dd = c.W.mid_dedup;
  const int64_t nm = BACK ? (dd ? c.W.status->n_own_b : c.W.status->n_mid_b)
                          : (dd ? c.W.status->n_own_a : c.W.status->n_mid_a);
  const uint32_t* lst = dd ? c.W.mid_own : c.W.mid_list;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b0 = blockIdx.x * (int64_t)blockDim.x + (threadIdx.x & ~31); b0 < nm; b0 += stride) {
    const int64_t i = b0 + lane;
    const bool valid = i < nm;
    int len = 0;
    int64_t p = 0;
    if (valid) {
      const int64_t k = BACK ? c.W.mid_cap - 1 - i : i;
      p = lst[2 * k];
      len = (int)lst[2 * k + 1];
    }
    const int wmax = BACK ? __reduce_max_sync(0xffffffffu, len) : 8;
    if (!valid) continue;
    constexpr int NB = BACK ? 16 : 8;
    uint8_t b[NB];
#pragma unroll
    for (int j = 0; j < NB; j++) b[j] = j < len ? gbyte(c, p + j) : 0;
    const int64_t G = c.gb + p;
    int32_t* dst = c.W.arena + G;
    int m;
    if constexpr (!BACK) m = merge_reg<8>(MT, b, len, dst);
    else m = wmax <= 12 ? merge_reg<12>(MT, b, len, dst) : merge_reg<16>(MT, b, len, dst);
    c.W.cnt[G] = (uint32_t)m;
    if (!dd) c.W.gsrc[G] = (uint32_t)G;
  }
}

// Offsets of an encode with no text: every segment is empty.
__global__ void k_empty_offsets(Call c, int64_t* out_offsets, int64_t* id_base) {
  const int64_t b = id_base ? id_base[0] : 0;
  for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s <= c.S; s += (int64_t)gridDim.x * blockDim.x)
    out_offsets[s] = b;
  if (id_base && blockIdx.x == 0 && threadIdx.x == 0) id_base[1] = b;
}

}  // namespace tk

// ============================================================================
// Host side.

using namespace tk;

static int cuda_fail(cudaError_t e, const char* what) {
  tk_set_error("%s: %s", what, cudaGetErrorString(e));
  return TK_E_CUDA;
}

#define TK_CUDA(call, what)                          \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// The mid-piece word cache pays for its table clear and extra launches from
// about this call size on (below it the side stream's latency, not its work,
// decides).
constexpr int64_t MID_DEDUP_MIN = 8ll << 20;
// Calls of at least this size merge their mid pieces (5..SHORT_MAX bytes) on
// a side stream with the mid-piece word cache, next to the tile kernel;
// smaller calls merge them inside the tile kernel (measured: the 256 MiB
// serving batch, whose requests repeat, is 0.57 ms faster per call with the
// word cache; the 4 MB agentic prompt and the 8 MiB multilingual text are
// 0.04-0.07 ms faster in the tile kernel).
constexpr int64_t MID_SIDE_MIN = 16ll << 20;

// Slots of the mid-piece word cache for a call of n bytes: one per 64 bytes
// (the serving batch repeats most words), at least 2^10, at most 2^22.
static uint32_t mtab_log2_for(int64_t n) {
  uint32_t l = 10;
  while (l < 22 && (1ll << l) < n / 64) l++;
  return l;
}

extern "C" int tk_workspace_create(const tk_tokenizer* tok, int64_t max_bytes, int64_t max_segments,
                                   tk_workspace** out) {
  if (!tok || !out || max_bytes < 0 || max_segments < 0) {
    tk_set_error("tk_workspace_create: bad argument");
    return TK_E_ARG;
  }
  *out = nullptr;
  if (max_bytes > (int64_t)PTOK_MASK - 1023) {  // positions (with batch padding) stay below 2^31
    tk_set_error("tk_workspace_create: max_bytes %lld above 2^31 - 1024", (long long)max_bytes);
    return TK_E_LIMIT;
  }
  tk_workspace* ws = new (std::nothrow) tk_workspace();
  if (!ws) return TK_E_NOMEM;
  ws->tok = tok;
  ws->device = tok->device;
  ws->num_sms = tok->num_sms;
  cudaSetDevice(tok->device);
  const int64_t nb = std::max<int64_t>(max_bytes, 1);
  // arrays indexed by global position: a pipelined call's batches sit up to
  // 16 bytes per batch (plus alignment) past their offset in the text
  const int64_t nbp = nb + 16 * (tk_workspace::PIPE_MAX + 2) + 2;
  const int64_t n_split_tiles = (nb + TILE - 1) / TILE + 1;
  const int64_t n_scan_tiles = (nb + 1 + SCAN_TILE - 1) / SCAN_TILE + 1;
  // bitmaps: the split writes whole tiles of the start bitmaps
  const int64_t cut_words = std::max<int64_t>((nb + 64) / 32 + 1, n_split_tiles * (TILE / 32) + 1);
  Work& w = ws->w;
  w.max_bytes = max_bytes;
  w.max_segments = max_segments;
  w.dtab_log2 = DTAB_LOG2;
  w.mid_cap = nb / MID_MIN + 2;
  w.mtab_log2_max = mtab_log2_for(nb);
  w.mtab_log2 = w.mtab_log2_max;
  struct Req { void** p; size_t bytes; };
  Req reqs[] = {
      {(void**)&w.status, sizeof(Status)},
      {(void**)&w.desc_a, sizeof(uint64_t) * n_split_tiles},
      {(void**)&w.desc_b, sizeof(uint64_t) * n_split_tiles},
      {(void**)&w.desc_w, sizeof(uint64_t) * n_split_tiles},
      {(void**)&w.desc_r, sizeof(uint64_t) * n_split_tiles},
      {(void**)&w.desc_c, sizeof(uint64_t) * n_scan_tiles},
      {(void**)&w.win_cut, sizeof(uint32_t) * cut_words},
      {(void**)&w.run_cut, sizeof(uint32_t) * cut_words},
      {(void**)&w.pbits, sizeof(uint32_t) * cut_words},
      {(void**)&w.sbits, sizeof(uint32_t) * cut_words},
      {(void**)&w.tile_first, sizeof(uint32_t) * n_split_tiles},
      {(void**)&w.cnt, sizeof(uint32_t) * nbp},
      {(void**)&w.offs, sizeof(uint32_t) * nbp},
      {(void**)&w.arena, sizeof(int32_t) * nbp},
      {(void**)&w.long_list, sizeof(uint32_t) * 2 * (nb / (SHORT_MAX + 1) + 2)},
      {(void**)&w.mid_list, sizeof(uint32_t) * 2 * (size_t)(nb / MID_MIN + 2)},
      {(void**)&w.mid_own, sizeof(uint32_t) * 2 * (size_t)(nb / MID_MIN + 2)},
      {(void**)&w.mtab, sizeof(unsigned long long) * 4 * ((size_t)1 << mtab_log2_for(nb))},
      {(void**)&w.staging, sizeof(uint32_t) * (size_t)(n_split_tiles * STG)},
      {(void**)&w.tile_count, sizeof(uint32_t) * (n_split_tiles + 1)},
      {(void**)&w.tile_base, sizeof(uint32_t) * (n_split_tiles + 2)},
      {(void**)&w.tile_meta, sizeof(uint32_t) * (n_split_tiles + 1)},
      {(void**)&w.seg_rel, sizeof(uint32_t) * (max_segments + 2)},
      {(void**)&w.tile_segs, sizeof(uint32_t) * 4 * (n_split_tiles + 1)},
      {(void**)&w.gsrc, sizeof(uint32_t) * nbp},
      {(void**)&w.dtab, sizeof(unsigned long long) * 2 * ((size_t)1 << DTAB_LOG2)},
      {(void**)&w.big_list, sizeof(uint32_t) * 2 * (nb / (MEDIUM_MAX + 1) + 2)},
      {(void**)&w.cl_list, sizeof(uint32_t) * 2 * (nb / (CLUSTER_MIN + 1) + 2)},
      {(void**)&w.lrk, sizeof(uint32_t) * nbp},
      {(void**)&w.lids2, sizeof(uint32_t) * nbp},
      {(void**)&w.lrk2, sizeof(uint32_t) * nbp},
      {(void**)&w.lsel, (size_t)nbp},
      {(void**)&w.lchg, (size_t)nbp},
      {(void**)&w.huge_list, sizeof(uint64_t) * 3 * (nb / HUGE_IDS + 2)},
      {(void**)&w.long_key, sizeof(uint64_t) * (nb / (SHORT_MAX + 1) + 2)},
      {(void**)&w.big_key, sizeof(uint64_t) * (nb / (MEDIUM_MAX + 1) + 2)},
      {(void**)&w.cl_key, sizeof(uint64_t) * (nb / (CLUSTER_MIN + 1) + 2)},
      {(void**)&ws->d_stage_text, (size_t)nb + 16 * (tk_workspace::PIPE_MAX + 2)},
      {(void**)&ws->d_stage_off, sizeof(int64_t) * (max_segments + 1 + tk_workspace::PIPE_MAX)},
      {(void**)&ws->d_stage_allow, (size_t)max_segments + 1},
      {(void**)&ws->d_stage_ids, sizeof(int32_t) * nb},
      {(void**)&ws->d_stage_offsets, sizeof(int64_t) * (max_segments + 1 + tk_workspace::PIPE_MAX)},
      {(void**)&ws->d_stage_raw, sizeof(int64_t) * (max_segments + 1 + tk_workspace::PIPE_MAX)},
      {(void**)&ws->d_pipe_base, sizeof(int64_t) * (tk_workspace::PIPE_MAX + 1)},
  };
  static_assert(sizeof(reqs) / sizeof(reqs[0]) <= tk_workspace::MAX_DEV, "workspace buffer table");
  for (auto& r : reqs) {
    cudaError_t e = cudaMalloc(r.p, r.bytes);
    if (e != cudaSuccess) {
      tk_set_error("tk_workspace_create: cudaMalloc(%zu): %s", r.bytes, cudaGetErrorString(e));
      tk_workspace_free(ws);
      return TK_E_NOMEM;
    }
    ws->dev_mem[ws->n_dev++] = *r.p;
  }
  if (cudaMallocHost((void**)&ws->h_status, sizeof(Status)) != cudaSuccess ||
      cudaMallocHost((void**)&ws->h_pipe_status, sizeof(Status) * tk_workspace::PIPE_MAX) != cudaSuccess) {
    tk_workspace_free(ws);
    tk_set_error("tk_workspace_create: cudaMallocHost failed");
    return TK_E_NOMEM;
  }
  int prio_lo = 0, prio_hi = 0;
  cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi);
  ws->prio_hi = prio_hi;
  bool ok = cudaStreamCreateWithFlags(&ws->s_h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&ws->s_d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithPriority(&ws->s_side, cudaStreamNonBlocking, prio_hi) == cudaSuccess &&
            cudaStreamCreateWithPriority(&ws->s_mid, cudaStreamNonBlocking, prio_hi) == cudaSuccess &&
            cudaStreamCreateWithPriority(&ws->s_cl, cudaStreamNonBlocking, prio_hi) == cudaSuccess &&
            cudaStreamCreateWithPriority(&ws->s_med, cudaStreamNonBlocking, prio_hi) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_dedup, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_cl, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_med, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_split, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_long, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_find, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_mid, cudaEventDisableTiming) == cudaSuccess &&
            cudaStreamCreateWithFlags(&ws->s_graph, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_gin, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&ws->ev_gout, cudaEventDisableTiming) == cudaSuccess;
  cudaEvent_t* evs[2 * tk_workspace::PIPE_MAX + 1];
  int ne = 0;
  evs[ne++] = &ws->ev_start;
  for (int k = 0; k < tk_workspace::PIPE_MAX; k++) {
    evs[ne++] = &ws->ev_h2d[k];
    evs[ne++] = &ws->ev_done[k];
  }
  for (int k = 0; k < ne && ok; k++) {
    ok = cudaEventCreateWithFlags(evs[k], cudaEventDisableTiming) == cudaSuccess;
    if (ok) ws->n_events = k + 1;
  }
  if (!ok) {
    tk_workspace_free(ws);
    tk_set_error("tk_workspace_create: stream or event creation failed");
    return TK_E_CUDA;
  }
  *out = ws;
  return TK_OK;
}

extern "C" void tk_workspace_free(tk_workspace* ws) {
  if (!ws) return;
  if (ws->s_h2d) cudaStreamSynchronize(ws->s_h2d);
  if (ws->s_d2h) cudaStreamSynchronize(ws->s_d2h);
  for (int i = 0; i < ws->n_dev; i++) cudaFree(ws->dev_mem[i]);
  if (ws->h_status) cudaFreeHost(ws->h_status);
  if (ws->h_pipe_status) cudaFreeHost(ws->h_pipe_status);
  // events in creation order: ev_start, then (ev_h2d[k], ev_done[k]) per batch
  for (int k = 0; k < ws->n_events; k++)
    cudaEventDestroy(k == 0 ? ws->ev_start : ((k - 1) % 2 == 0 ? ws->ev_h2d[(k - 1) / 2] : ws->ev_done[(k - 1) / 2]));
  if (ws->s_side) cudaStreamSynchronize(ws->s_side);
  if (ws->s_mid) cudaStreamSynchronize(ws->s_mid);
  if (ws->s_cl) cudaStreamSynchronize(ws->s_cl);
  if (ws->s_med) cudaStreamSynchronize(ws->s_med);
  if (ws->ev_dedup) cudaEventDestroy(ws->ev_dedup);
  if (ws->ev_cl) cudaEventDestroy(ws->ev_cl);
  if (ws->ev_med) cudaEventDestroy(ws->ev_med);
  if (ws->s_cl) cudaStreamDestroy(ws->s_cl);
  if (ws->s_med) cudaStreamDestroy(ws->s_med);
  if (ws->ev_split) cudaEventDestroy(ws->ev_split);
  if (ws->ev_long) cudaEventDestroy(ws->ev_long);
  if (ws->ev_find) cudaEventDestroy(ws->ev_find);
  if (ws->ev_mid) cudaEventDestroy(ws->ev_mid);
  if (ws->s_h2d) cudaStreamDestroy(ws->s_h2d);
  if (ws->s_d2h) cudaStreamDestroy(ws->s_d2h);
  if (ws->s_side) cudaStreamDestroy(ws->s_side);
  if (ws->s_mid) cudaStreamDestroy(ws->s_mid);
  if (ws->s_graph) cudaStreamSynchronize(ws->s_graph);
  if (ws->g_exec) cudaGraphExecDestroy(ws->g_exec);
  if (ws->ev_gin) cudaEventDestroy(ws->ev_gin);
  if (ws->ev_gout) cudaEventDestroy(ws->ev_gout);
  if (ws->s_graph) cudaStreamDestroy(ws->s_graph);
  delete ws;
}

// Launches the whole encode on `st`; the status block stays on the device.
// id_base: null, or a pipelined batch's slot (see k_seg_offsets).
static int encode_launch(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* d_text, int64_t n,
                         const int64_t* d_seg_off, const uint8_t* d_allow, int64_t S, int safe,
                         int32_t* d_out, int64_t cap, int64_t* d_out_offsets, int64_t* id_base,
                         int64_t gb, cudaStream_t st) {
  Call c;
  c.text = d_text;
  c.n = n;
  c.gb = gb;
  c.seg_off = d_seg_off;
  c.allow = d_allow;
  c.S = S;
  c.safe = safe ? 1 : 0;
  c.T = tok->t;
  c.W = ws->w;
  c.W.mtab_log2 = std::min(mtab_log2_for(n), ws->w.mtab_log2_max);
  c.W.mid_side = n >= MID_SIDE_MIN ? 1 : 0;
  c.W.mid_dedup = (c.W.mid_side && n >= MID_DEDUP_MIN) ? 1 : 0;
  c.W.use_cache = ws->cache ? 1 : 0;
  if (ws->cache) c.W.cache = ws->cache->d;
  const int64_t n_split_tiles = (n + TILE - 1) / TILE;
  const int64_t n_scan_tiles = (n + 1 + SCAN_TILE - 1) / SCAN_TILE + 1;
  const int64_t cut_words = (n + 64) / 32 + 1;
  const int sms = ws->num_sms;
  const int seg_grid = (int)std::max<int64_t>(1, std::min<int64_t>((S + 256) / 256, (int64_t)sms * 4));
  tk_prof_mark(ws, "k_reset", st);
  k_reset<<<sms * 2, 256, 0, st>>>(c.W, n_split_tiles + 1, n_scan_tiles, c.safe, cut_words,
                                   n_split_tiles, gb == 0 ? 1 : 0);
  tk_prof_mark(ws, "k_check_segments", st);
  k_check_segments<<<seg_grid, 256, 0, st>>>(c);
  if (n > 0) {
    if (ws->split_per_sm == 0) {  // once per workspace: launch shapes and shared-memory limits
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ws->split_per_sm, k_split, SPLIT_THREADS, 0);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ws->scan_per_sm, k_chunk_scan, SPLIT_THREADS, 0);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ws->copy_per_sm, k_copy_out, COPY_THREADS, 0);
      TK_CUDA(cudaFuncSetAttribute(k_merge_big, cudaFuncAttributeMaxDynamicSharedMemorySize, BIG_SMEM),
              "smem attribute");
      TK_CUDA(cudaFuncSetAttribute(k_encode_tiles<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)sizeof(EncSmem)), "smem attribute");
      TK_CUDA(cudaFuncSetAttribute(k_encode_tiles<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)sizeof(EncSmem)), "smem attribute");
      ws->split_per_sm = std::max(ws->split_per_sm, 1);
      ws->scan_per_sm = std::max(ws->scan_per_sm, 1);
      ws->copy_per_sm = std::max(ws->copy_per_sm, 1);
    }
    const int split_grid = (int)std::min<int64_t>(n_split_tiles, (int64_t)sms * ws->split_per_sm);
    const int scan_grid = (int)std::min<int64_t>(n_split_tiles, (int64_t)sms * ws->scan_per_sm);
    tk_prof_mark(ws, "k_tile_segs", st);
    k_tile_segs<<<(int)std::min<int64_t>((4 * n_split_tiles + 255) / 256, (int64_t)sms * 8), 256, 0, st>>>(c);
    if (c.safe) {
      tk_prof_mark(ws, "k_chunk_scan_windows", st);
      k_chunk_scan<<<scan_grid, SPLIT_THREADS, 0, st>>>(c, 0);
      tk_prof_mark(ws, "k_chunk_scan_runs", st);
      k_chunk_scan<<<scan_grid, SPLIT_THREADS, 0, st>>>(c, 1);
    }
    tk_prof_mark(ws, "k_split", st);
    k_split<<<split_grid, SPLIT_THREADS, 0, st>>>(c);
    // The long pieces (listing, word cache, merges) run on a second stream
    // next to the tile kernel, which needs their counts only in k_long_fixup.
    cudaStream_t side = ws->s_side;
    TK_CUDA(cudaEventRecord(ws->ev_split, st), "fork");
    TK_CUDA(cudaStreamWaitEvent(side, ws->ev_split, 0), "fork");
    tk_prof_mark(ws, "k_find_long", side);
    k_find_long<<<(int)std::min<int64_t>((n_split_tiles * (TILE / 32 / FIND_WPT) + 255) / 256, (int64_t)sms * 16), 256, 0, side>>>(c);
    // the mid pieces of large calls on a third stream, next to the long
    // pieces' chain
    cudaStream_t mid = ws->s_mid;
    if (c.W.mid_side) {
      TK_CUDA(cudaEventRecord(ws->ev_find, side), "fork");
      TK_CUDA(cudaStreamWaitEvent(mid, ws->ev_find, 0), "fork");
      if (c.W.mid_dedup) {
        tk_prof_mark(ws, "k_clear_mtab", mid);
        k_clear_mtab<<<sms * 4, 256, 0, mid>>>(c.W);
        tk_prof_mark(ws, "k_dedup_mid", mid);
        k_dedup_mid<false><<<sms * 8, ETHREADS, 0, mid>>>(c);
        k_dedup_mid<true><<<sms * 4, ETHREADS, 0, mid>>>(c);
      }
      tk_prof_mark(ws, "k_merge_mid", mid);
      k_merge_mid<false><<<sms * 8, ETHREADS, 0, mid>>>(c);
      tk_prof_mark(ws, "k_merge_mid_long", mid);
      k_merge_mid<true><<<sms * 4, ETHREADS, 0, mid>>>(c);
      tk_prof_mark(ws, nullptr, mid);
      TK_CUDA(cudaEventRecord(ws->ev_mid, mid), "join");
    }
    tk_prof_mark(ws, "k_dedup_medium", side);
    k_dedup_medium<<<sms * 8, ETHREADS, 0, side>>>(c);
    tk_prof_mark(ws, "k_dedup_big", side);
    k_dedup_big<<<sms, 1024, 0, side>>>(c);
    if (c.W.use_cache) {
      tk_prof_mark(ws, "k_cache_lookup", side);
      k_cache_lookup<<<sms * 8, ETHREADS, 0, side>>>(c);
      tk_prof_mark(ws, "k_cache_lookup_big", side);
      k_cache_lookup_big<<<sms, 1024, 0, side>>>(c);
    }
    // the three merge tiers take disjoint lists: the cluster and medium
    // merges run on streams of their own next to the big merges
    TK_CUDA(cudaEventRecord(ws->ev_dedup, side), "fork");
    TK_CUDA(cudaStreamWaitEvent(ws->s_cl, ws->ev_dedup, 0), "fork");
    TK_CUDA(cudaStreamWaitEvent(ws->s_med, ws->ev_dedup, 0), "fork");
    tk_prof_mark(ws, "k_merge_cluster", ws->s_cl);
    k_merge_cluster<<<MERGE_CL * std::max(1, sms / MERGE_CL), CL_THREADS, 0, ws->s_cl>>>(c);
    tk_prof_mark(ws, nullptr, ws->s_cl);
    TK_CUDA(cudaEventRecord(ws->ev_cl, ws->s_cl), "join");
    tk_prof_mark(ws, "k_merge_medium", ws->s_med);
    k_merge_medium<<<sms * 4, ETHREADS, 0, ws->s_med>>>(c);
    tk_prof_mark(ws, nullptr, ws->s_med);
    TK_CUDA(cudaEventRecord(ws->ev_med, ws->s_med), "join");
    tk_prof_mark(ws, "k_merge_big", side);
    k_merge_big<<<sms, BIG_THREADS, BIG_SMEM, side>>>(c);
    tk_prof_mark(ws, nullptr, side);
    TK_CUDA(cudaStreamWaitEvent(side, ws->ev_cl, 0), "join");
    TK_CUDA(cudaStreamWaitEvent(side, ws->ev_med, 0), "join");
    if (c.W.use_cache) {
      tk_prof_mark(ws, "k_cache_insert", side);
      k_cache_insert<<<sms * 8, ETHREADS, 0, side>>>(c);
    }
    tk_prof_mark(ws, nullptr, side);
    TK_CUDA(cudaEventRecord(ws->ev_long, side), "join");
    tk_prof_mark(ws, "k_encode_tiles", st);
    if (c.W.mid_side) k_encode_tiles<false><<<(int)n_split_tiles, ETHREADS, sizeof(EncSmem), st>>>(c);
    else k_encode_tiles<true><<<(int)n_split_tiles, ETHREADS, sizeof(EncSmem), st>>>(c);
    tk_prof_mark(ws, nullptr, st);
    TK_CUDA(cudaStreamWaitEvent(st, ws->ev_long, 0), "join");
    if (c.W.mid_side) TK_CUDA(cudaStreamWaitEvent(st, ws->ev_mid, 0), "join");
    tk_prof_mark(ws, "k_long_fixup", st);
    k_long_fixup<<<(int)std::min<int64_t>((n_split_tiles * 32 + ETHREADS - 1) / ETHREADS, (int64_t)sms * 8), ETHREADS, 0, st>>>(c);
    tk_prof_mark(ws, "k_scan_u32", st);
    int rc = tk_scan_u32(ws, ws->w.tile_count, ws->w.tile_base, &ws->w.status->n_tiles, n_split_tiles, 3, st);
    if (rc) return rc;
    tk_prof_mark(ws, "k_copy_out", st);
    k_copy_out<<<(int)std::min<int64_t>(n_split_tiles, (int64_t)sms * ws->copy_per_sm), COPY_THREADS, 0,
                 st>>>(c, d_out, cap);
    tk_prof_mark(ws, "k_copy_huge", st);
    k_copy_huge<<<sms * 4, ETHREADS, 0, st>>>(c, d_out, cap);
    tk_prof_mark(ws, "k_seg_offsets", st);
    k_seg_offsets<<<seg_grid, 256, 0, st>>>(c, d_out_offsets, id_base);
  } else {
    tk_prof_mark(ws, "k_empty_offsets", st);
    k_empty_offsets<<<seg_grid, 256, 0, st>>>(c, d_out_offsets, id_base);
  }
  tk_prof_mark(ws, nullptr, st);
  TK_CUDA(cudaGetLastError(), "encode launch");
  return TK_OK;
}

// The outcome recorded in a status block; pos_base shifts error positions
// (a pipelined batch's first byte).
static int encode_result(const Status& hs, int64_t cap, int64_t pos_base) {
  if (hs.code == TK_E_UTF8) {
    tk_set_error("invalid UTF-8 at byte %lld", (long long)(hs.err_pos + pos_base));
    return TK_E_UTF8;
  }
  if (hs.code) {
    tk_set_error("encode failed on the device (code %d, site %d)", hs.code, hs.err_kind);
    return hs.code;
  }
  if (hs.n_ids > cap) {
    tk_set_error("output capacity %lld < %lld ids", (long long)cap, (long long)hs.n_ids);
    return TK_E_CAPACITY;
  }
  return TK_OK;
}

// A captured graph's kernel nodes keep no stream priority: the kernels that
// run on the side streams (long and mid pieces) get the side streams' high
// priority back, so that they are not starved by the tile kernel's CTAs.
static void graph_side_priority(cudaGraph_t g, int prio) {
  const void* side[] = {(const void*)k_find_long, (const void*)k_clear_mtab, (const void*)k_dedup_mid<false>,
                        (const void*)k_dedup_mid<true>, (const void*)k_merge_mid<false>,
                        (const void*)k_merge_mid<true>, (const void*)k_dedup_medium, (const void*)k_dedup_big,
                        (const void*)k_cache_lookup, (const void*)k_cache_lookup_big,
                        (const void*)k_merge_cluster, (const void*)k_merge_medium, (const void*)k_merge_big,
                        (const void*)k_cache_insert};
  size_t nn = 0;
  if (cudaGraphGetNodes(g, nullptr, &nn) != cudaSuccess || nn == 0) return;
  std::vector<cudaGraphNode_t> nodes(nn);
  if (cudaGraphGetNodes(g, nodes.data(), &nn) != cudaSuccess) return;
  for (cudaGraphNode_t node : nodes) {
    cudaGraphNodeType t;
    cudaKernelNodeParams kp;
    if (cudaGraphNodeGetType(node, &t) != cudaSuccess || t != cudaGraphNodeTypeKernel) continue;
    if (cudaGraphKernelNodeGetParams(node, &kp) != cudaSuccess) continue;
    for (const void* f : side)
      if (kp.func == f) {
        cudaLaunchAttributeValue v = {};
        v.priority = prio;
        cudaGraphKernelNodeSetAttribute(node, cudaLaunchAttributePriority, &v);
        break;
      }
  }
  cudaGetLastError();
}

// Launches the whole encode on `st` and reads back the status (one sync).  A
// call under MID_SIDE_MIN bytes repeated with the same arguments is captured
// into a graph the second time (on the workspace's graph stream, joined with
// `st` by events) and replayed from then on: one launch instead of about
// thirty, with the kernels' parameters unchanged (every call starts by
// resetting its state on the device).  Larger calls (whose kernels are long
// next to their launches; replayed, the 256 MiB serving batch measured 2.97
// instead of 2.88 ms), profiled calls and failed captures launch directly.
static int encode_device(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* d_text, int64_t n,
                         const int64_t* d_seg_off, const uint8_t* d_allow, int64_t S, int safe,
                         int32_t* d_out, int64_t cap, int64_t* d_out_offsets, int64_t* h_n_ids,
                         cudaStream_t st) {
  const uint64_t key[12] = {(uint64_t)(uintptr_t)tok, (uint64_t)(uintptr_t)d_text, (uint64_t)n,
                            (uint64_t)(uintptr_t)d_seg_off, (uint64_t)(uintptr_t)d_allow, (uint64_t)S,
                            (uint64_t)safe, (uint64_t)(uintptr_t)d_out, (uint64_t)cap,
                            (uint64_t)(uintptr_t)d_out_offsets, (uint64_t)(uintptr_t)ws->cache, 0};
  if (ws->g_seen == 0 || memcmp(key, ws->g_key, sizeof(key)) != 0) {
    if (ws->g_exec) {
      cudaGraphExecDestroy(ws->g_exec);
      ws->g_exec = nullptr;
    }
    memcpy(ws->g_key, key, sizeof(key));
    ws->g_seen = 0;
  }
  ws->g_seen++;
  cudaStream_t run = st;
  if (!ws->prof.on && !ws->g_off && ws->g_seen >= 2 && n > 0 && n < MID_SIDE_MIN) {
    TK_CUDA(cudaEventRecord(ws->ev_gin, st), "graph join");
    TK_CUDA(cudaStreamWaitEvent(ws->s_graph, ws->ev_gin, 0), "graph join");
    if (!ws->g_exec) {
      cudaGraph_t g = nullptr;
      int rc = TK_E_CUDA;
      if (cudaStreamBeginCapture(ws->s_graph, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        rc = encode_launch(tok, ws, d_text, n, d_seg_off, d_allow, S, safe, d_out, cap, d_out_offsets,
                           nullptr, 0, ws->s_graph);
        const cudaError_t e = cudaStreamEndCapture(ws->s_graph, &g);
        if (rc == TK_OK && e == cudaSuccess && g) graph_side_priority(g, ws->prio_hi);
        if (rc == TK_OK && (e != cudaSuccess || !g || cudaGraphInstantiate(&ws->g_exec, g, 0) != cudaSuccess)) {
          ws->g_exec = nullptr;
          rc = TK_E_CUDA;
        }
      }
      if (g) cudaGraphDestroy(g);
      if (!ws->g_exec) {
        ws->g_off = 1;  // launch directly from now on
        cudaGetLastError();
      }
    }
    if (ws->g_exec) {
      TK_CUDA(cudaGraphLaunch(ws->g_exec, ws->s_graph), "graph launch");
      run = ws->s_graph;
    }
  }
  if (run == st) {
    int rc = encode_launch(tok, ws, d_text, n, d_seg_off, d_allow, S, safe, d_out, cap, d_out_offsets,
                           nullptr, 0, st);
    if (rc) return rc;
  }
  TK_CUDA(cudaMemcpyAsync(ws->h_status, ws->w.status, sizeof(Status), cudaMemcpyDeviceToHost, run),
          "status copy");
  if (run != st) {
    TK_CUDA(cudaEventRecord(ws->ev_gout, run), "graph join");
    TK_CUDA(cudaStreamWaitEvent(st, ws->ev_gout, 0), "graph join");
  }
  TK_CUDA(cudaStreamSynchronize(run), "encode");
  tk_prof_finish(ws, st);
  if (h_n_ids) *h_n_ids = ws->h_status->n_ids;
  return encode_result(*ws->h_status, cap, 0);
}

extern "C" int tk_last_cache_stats(const tk_workspace* ws, int64_t* hits, int64_t* inserts) {
  if (!ws) return TK_E_ARG;
  if (hits) *hits = ws->h_status->n_cache_hits;
  if (inserts) *inserts = ws->h_status->n_cache_inserts;
  return TK_OK;
}

extern "C" int tk_last_stats(const tk_workspace* ws, int64_t* n_pretokens, int64_t* n_ids,
                             int64_t* n_long) {
  if (!ws) return TK_E_ARG;
  if (n_pretokens) *n_pretokens = ws->h_status->n_ptok;
  if (n_ids) *n_ids = ws->h_status->n_ids;
  if (n_long) *n_long = ws->h_status->n_long;
  return TK_OK;
}

static int check_encode_args(const tk_tokenizer* tok, tk_workspace* ws, const void* text, int64_t n,
                             const void* seg_off, const void* allow, int64_t S, const void* out,
                             int64_t cap, const void* out_off) {
  if (!tok || !ws || ws->tok != tok || n < 0 || S < 0 || cap < 0 || !seg_off || !out_off ||
      (n > 0 && !text) || (S > 0 && !allow) || (cap > 0 && !out)) {
    tk_set_error("tk_encode_segments: bad argument");
    return TK_E_ARG;
  }
  if (n > ws->w.max_bytes || S > ws->w.max_segments) {
    tk_set_error("tk_encode_segments: %lld bytes / %lld segments above the workspace limits %lld / %lld",
                 (long long)n, (long long)S, (long long)ws->w.max_bytes, (long long)ws->w.max_segments);
    return TK_E_LIMIT;
  }
  if (S == 0 && n != 0) {
    tk_set_error("tk_encode_segments: text without segments");
    return TK_E_ARG;
  }
  return TK_OK;
}

extern "C" int tk_encode_segments(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* d_text,
                                  int64_t n_bytes, const int64_t* d_seg_off,
                                  const uint8_t* d_allow_special, int64_t S, int tiktoken_safe,
                                  int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                                  int64_t* h_n_ids, void* cuda_stream) {
  int rc = check_encode_args(tok, ws, d_text, n_bytes, d_seg_off, d_allow_special, S, d_out_ids,
                             out_capacity, d_out_offsets);
  if (rc) return rc;
  cudaSetDevice(ws->device);
  return encode_device(tok, ws, d_text, n_bytes, d_seg_off, d_allow_special, S, tiktoken_safe,
                       d_out_ids, out_capacity, d_out_offsets, h_n_ids, (cudaStream_t)cuda_stream);
}

// Batches of a pipelined host call: consecutive segments, about PIPE_TARGET
// bytes each (at least PIPE_MIN_BYTES), at most PIPE_MAX batches.  Returns
// the batch count (1: no pipelining) and fills first[k] = the first segment
// of batch k, first[count] = S.  Offsets that are not a valid table give 1:
// the one-batch call then reports the error from the device check.
constexpr int64_t PIPE_MIN_BYTES = 16ll << 20;
// Start of batch k's text in the staging buffer: 16-byte aligned, after the
// end of batch k - 1's (which ends below b0 + 16 k).
static int64_t pipe_text_at(int64_t b0, int k) { return (b0 + 16 * (int64_t)k + 15) & ~(int64_t)15; }
constexpr int PIPE_TARGET = 8;
static int plan_batches(const int64_t* seg_off, int64_t S, int64_t n, int64_t* first) {
  if (S < 2 || n < 2 * PIPE_MIN_BYTES || seg_off[0] != 0 || seg_off[S] != n) return 1;
  for (int64_t s = 0; s < S; s++)
    if (seg_off[s + 1] < seg_off[s]) return 1;
  const int64_t target = std::max<int64_t>(PIPE_MIN_BYTES, (n + PIPE_TARGET - 1) / PIPE_TARGET);
  int k = 0;
  first[0] = 0;
  for (int64_t s = 0; s < S; s++) {
    // close the batch before segment s when it already holds `target` bytes
    if (s > first[k] && seg_off[s] - seg_off[first[k]] >= target && k + 1 < tk_workspace::PIPE_MAX)
      first[++k] = s;
  }
  first[k + 1] = S;
  return k + 1;
}

extern "C" int tk_encode_segments_host(const tk_tokenizer* tok, tk_workspace* ws, const uint8_t* h_text,
                                       int64_t n_bytes, const int64_t* h_seg_off,
                                       const uint8_t* h_allow_special, int64_t S, int tiktoken_safe,
                                       int32_t* h_out_ids, int64_t out_capacity, int64_t* h_out_offsets,
                                       int64_t* h_n_ids, void* cuda_stream) {
  int rc = check_encode_args(tok, ws, h_text, n_bytes, h_seg_off, h_allow_special, S, h_out_ids,
                             out_capacity, h_out_offsets);
  if (rc) return rc;
  cudaSetDevice(ws->device);
  cudaStream_t st = (cudaStream_t)cuda_stream;
  int64_t first[tk_workspace::PIPE_MAX + 1];
  const int nbat = ws->prof.on ? 1 : plan_batches(h_seg_off, S, n_bytes, first);
  if (nbat == 1) {
    if (n_bytes) TK_CUDA(cudaMemcpyAsync(ws->d_stage_text, h_text, n_bytes, cudaMemcpyHostToDevice, st), "h2d text");
    TK_CUDA(cudaMemcpyAsync(ws->d_stage_off, h_seg_off, sizeof(int64_t) * (S + 1), cudaMemcpyHostToDevice, st),
            "h2d offsets");
    if (S) TK_CUDA(cudaMemcpyAsync(ws->d_stage_allow, h_allow_special, S, cudaMemcpyHostToDevice, st), "h2d allow");
    const int64_t dcap = std::min<int64_t>(out_capacity, std::max<int64_t>(ws->w.max_bytes, 1));
    int64_t n_ids = 0;
    rc = encode_device(tok, ws, ws->d_stage_text, n_bytes, ws->d_stage_off, ws->d_stage_allow, S,
                       tiktoken_safe, ws->d_stage_ids, dcap, ws->d_stage_offsets, &n_ids, st);
    if (h_n_ids) *h_n_ids = n_ids;
    if (rc) return rc;
    if (n_ids) TK_CUDA(cudaMemcpyAsync(h_out_ids, ws->d_stage_ids, sizeof(int32_t) * n_ids, cudaMemcpyDeviceToHost, st),
                       "d2h ids");
    TK_CUDA(cudaMemcpyAsync(h_out_offsets, ws->d_stage_offsets, sizeof(int64_t) * (S + 1), cudaMemcpyDeviceToHost, st),
            "d2h offsets");
    TK_CUDA(cudaStreamSynchronize(st), "encode (host buffers)");
    return TK_OK;
  }
  // Pipelined: batch k's bytes, segment offsets, flags and ids sit in
  // disjoint parts of the staging buffers (text and ids at the batch's byte
  // offset, offsets at first[k] + k).  All copies in go first on s_h2d; the
  // encodes run in order on st; batch k's ids go out on s_d2h while batch
  // k + 1 encodes.  The workspace's other buffers serve one batch at a time,
  // in stream order.
  TK_CUDA(cudaEventRecord(ws->ev_start, st), "pipeline start");
  TK_CUDA(cudaStreamWaitEvent(ws->s_h2d, ws->ev_start, 0), "pipeline start");
  TK_CUDA(cudaStreamWaitEvent(ws->s_d2h, ws->ev_start, 0), "pipeline start");
  TK_CUDA(cudaMemsetAsync(ws->d_pipe_base, 0, sizeof(int64_t), st), "pipeline base");
  for (int k = 0; k < nbat; k++) {
    const int64_t s0 = first[k], s1 = first[k + 1], b0 = h_seg_off[s0], b1 = h_seg_off[s1];
    if (b1 > b0)
      TK_CUDA(cudaMemcpyAsync(ws->d_stage_text + pipe_text_at(b0, k), h_text + b0, b1 - b0,
                              cudaMemcpyHostToDevice, ws->s_h2d), "h2d text");
    TK_CUDA(cudaMemcpyAsync(ws->d_stage_raw + s0 + k, h_seg_off + s0, sizeof(int64_t) * (s1 - s0 + 1),
                            cudaMemcpyHostToDevice, ws->s_h2d), "h2d offsets");
    TK_CUDA(cudaMemcpyAsync(ws->d_stage_allow + s0, h_allow_special + s0, s1 - s0, cudaMemcpyHostToDevice,
                            ws->s_h2d), "h2d allow");
    TK_CUDA(cudaEventRecord(ws->ev_h2d[k], ws->s_h2d), "h2d event");
  }
  for (int k = 0; k < nbat; k++) {
    const int64_t s0 = first[k], s1 = first[k + 1], b0 = h_seg_off[s0], b1 = h_seg_off[s1];
    TK_CUDA(cudaStreamWaitEvent(st, ws->ev_h2d[k], 0), "h2d wait");
    k_rebase<<<(int)std::min<int64_t>((s1 - s0 + 256) / 256, 64), 256, 0, st>>>(
        ws->d_stage_raw + s0 + k, ws->d_stage_off + s0 + k, s1 - s0 + 1);
    rc = encode_launch(tok, ws, ws->d_stage_text + pipe_text_at(b0, k), b1 - b0, ws->d_stage_off + s0 + k,
                       ws->d_stage_allow + s0, s1 - s0, tiktoken_safe, ws->d_stage_ids + b0,
                       std::max<int64_t>(b1 - b0, 0), ws->d_stage_offsets + s0 + k, ws->d_pipe_base + k,
                       pipe_text_at(b0, k), st);
    if (rc) {
      cudaStreamSynchronize(st);
      cudaStreamSynchronize(ws->s_h2d);
      cudaStreamSynchronize(ws->s_d2h);
      return rc;
    }
    TK_CUDA(cudaMemcpyAsync(&ws->h_pipe_status[k], ws->w.status, sizeof(Status), cudaMemcpyDeviceToHost, st),
            "status copy");
    TK_CUDA(cudaEventRecord(ws->ev_done[k], st), "batch event");
  }
  // Copies out, batch by batch as each ends (the ids' count is known once the
  // batch's status arrives).  Everything on s_d2h is enqueued here, after the
  // host saw the batch end, so no copy waits behind a later batch.
  int first_rc = TK_OK;
  int64_t total = 0;
  Status sum = {};
  for (int k = 0; k < nbat; k++) {
    TK_CUDA(cudaEventSynchronize(ws->ev_done[k]), "batch");
    const Status& hs = ws->h_pipe_status[k];
    const int64_t s0 = first[k], s1 = first[k + 1];
    const int64_t b0 = h_seg_off[s0], b1 = h_seg_off[s1];
    TK_CUDA(cudaMemcpyAsync(h_out_offsets + s0, ws->d_stage_offsets + s0 + k,
                            sizeof(int64_t) * (s1 - s0 + (k == nbat - 1 ? 1 : 0)), cudaMemcpyDeviceToHost,
                            ws->s_d2h), "d2h offsets");
    const int brc = encode_result(hs, std::max<int64_t>(b1 - b0, 0), b0);
    if (brc && !first_rc) first_rc = brc;
    sum.n_ptok += hs.n_ptok;
    sum.n_long += hs.n_long;
    sum.n_cache_hits += hs.n_cache_hits;
    sum.n_cache_inserts += hs.n_cache_inserts;
    if (!first_rc && hs.n_ids && total + hs.n_ids <= out_capacity)
      TK_CUDA(cudaMemcpyAsync(h_out_ids + total, ws->d_stage_ids + b0, sizeof(int32_t) * hs.n_ids,
                              cudaMemcpyDeviceToHost, ws->s_d2h), "d2h ids");
    total += hs.n_ids;
  }
  TK_CUDA(cudaStreamSynchronize(ws->s_d2h), "encode (host buffers)");
  TK_CUDA(cudaStreamSynchronize(st), "encode (host buffers)");
  sum.n_ids = total;
  *ws->h_status = sum;
  if (h_n_ids) *h_n_ids = total;
  if (first_rc) return first_rc;
  if (total > out_capacity) {
    tk_set_error("output capacity %lld < %lld ids", (long long)out_capacity, (long long)total);
    return TK_E_CAPACITY;
  }
  return TK_OK;
}

// --------------------------------------------------------------------------
// Cross-call word cache: host API.
extern "C" int tk_cache_create(const tk_tokenizer* tok, int64_t max_bytes, tk_cache** out) {
  using namespace tk;
  if (!tok || !out || max_bytes < SHORT_MAX + 1) {
    tk_set_error("tk_cache_create: bad argument (max_bytes must be at least %d)", SHORT_MAX + 1);
    return TK_E_ARG;
  }
  *out = nullptr;
  tk_cache* cc = new (std::nothrow) tk_cache();
  if (!cc) return TK_E_NOMEM;
  cc->tok = tok;
  cc->device = tok->device;
  cudaSetDevice(tok->device);
  CacheDev& d = cc->d;
  d.max_bytes = (uint64_t)max_bytes;
  d.max_ids = (uint64_t)max_bytes;  // a piece never has more ids than bytes
  d.max_entries = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)max_bytes / (SHORT_MAX + 1), 1ull << 24));
  d.slot_log2 = 4;
  while ((1ull << d.slot_log2) < 2 * d.max_entries) d.slot_log2++;
  struct Req { void** p; size_t bytes; };
  Req reqs[] = {
      {(void**)&d.slots, sizeof(unsigned long long) * 2 * ((size_t)1 << d.slot_log2)},
      {(void**)&d.entries, sizeof(CacheEntry) * (size_t)d.max_entries},
      {(void**)&d.bytes, (size_t)d.max_bytes},
      {(void**)&d.ids, sizeof(int32_t) * (size_t)d.max_ids},
      {(void**)&d.used, sizeof(unsigned long long) * 3},
  };
  static_assert(sizeof(reqs) / sizeof(reqs[0]) <= tk_cache::MAX_DEV, "cache buffer table");
  for (auto& r : reqs) {
    if (cudaMalloc(r.p, r.bytes) != cudaSuccess) {
      tk_set_error("tk_cache_create: cudaMalloc(%zu) failed", r.bytes);
      tk_cache_free(cc);
      return TK_E_NOMEM;
    }
    cc->dev_mem[cc->n_dev++] = *r.p;
  }
  if (cudaMemset(d.slots, 0, sizeof(unsigned long long) * 2 * ((size_t)1 << d.slot_log2)) != cudaSuccess ||
      cudaMemset(d.used, 0, sizeof(unsigned long long) * 3) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    tk_set_error("tk_cache_create: clearing the cache failed");
    tk_cache_free(cc);
    return TK_E_CUDA;
  }
  *out = cc;
  return TK_OK;
}

extern "C" void tk_cache_free(tk_cache* cc) {
  if (!cc) return;
  for (int i = 0; i < cc->n_dev; i++) cudaFree(cc->dev_mem[i]);
  delete cc;
}

extern "C" int tk_cache_clear(tk_cache* cc, void* cuda_stream) {
  if (!cc) return TK_E_ARG;
  cudaSetDevice(cc->device);
  cudaStream_t st = (cudaStream_t)cuda_stream;
  cudaError_t e = cudaMemsetAsync(cc->d.slots, 0, sizeof(unsigned long long) * 2 * ((size_t)1 << cc->d.slot_log2), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(cc->d.used, 0, sizeof(unsigned long long) * 3, st);
  if (e != cudaSuccess) {
    tk_set_error("tk_cache_clear: %s", cudaGetErrorString(e));
    return TK_E_CUDA;
  }
  return TK_OK;
}

extern "C" int tk_cache_stats(const tk_cache* cc, int64_t* n_entries, int64_t* bytes_used, int64_t* ids_used) {
  if (!cc) return TK_E_ARG;
  cudaSetDevice(cc->device);
  unsigned long long u[3] = {0, 0, 0};
  if (cudaMemcpy(u, cc->d.used, sizeof(u), cudaMemcpyDeviceToHost) != cudaSuccess) {
    tk_set_error("tk_cache_stats: copy failed");
    return TK_E_CUDA;
  }
  // reservations past the capacity did not take effect
  if (n_entries) *n_entries = (int64_t)std::min<unsigned long long>(u[0], cc->d.max_entries);
  if (bytes_used) *bytes_used = (int64_t)std::min<unsigned long long>(u[1], cc->d.max_bytes);
  if (ids_used) *ids_used = (int64_t)std::min<unsigned long long>(u[2], cc->d.max_ids);
  return TK_OK;
}

extern "C" int tk_workspace_set_cache(tk_workspace* ws, tk_cache* cc) {
  if (!ws || (cc && cc->tok != ws->tok)) {
    tk_set_error("tk_workspace_set_cache: the cache belongs to another tokenizer");
    return TK_E_ARG;
  }
  ws->cache = cc;
  return TK_OK;
}
