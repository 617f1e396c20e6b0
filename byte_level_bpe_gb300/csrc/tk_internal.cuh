// tk_internal.cuh -- definitions shared by the libtk translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "tk.h"

namespace tk {

constexpr uint32_t RANK_MAX = 0xFFFFFFFFu;
constexpr uint32_t MAX_ID = (1u << 20) - 2;  // ids and ranks fit the packed pair slots
constexpr int MAX_SPECIAL = 64;               // longest special string, bytes
constexpr int MAX_SPECIALS = 256;

// Split tiles: 4 KiB of text per tile, 256 threads, 16 bytes per thread.  The
// tile is loaded with HALO bytes on each side; piece starts (segment starts,
// safe-chunking cuts, special spans) are exact for positions at least TRUST
// bytes inside the loaded window (a special of up to 64 bytes must fit).
constexpr int TILE = 4096;
constexpr int SPLIT_THREADS = 256;
constexpr int HALO = 128;
constexpr int TRUST = 64;
constexpr int WIN = TILE + 2 * HALO;

constexpr int SHORT_MAX = 16;   // pre-tokens up to this length merge one per thread
constexpr int MID_MIN = 5;      // ... those of MID_MIN..SHORT_MAX bytes over the whole grid
                                // (k_merge_mid), the shorter ones inside the tile kernel
constexpr int SCAN_THREADS = 256;
constexpr int SCAN_ITEMS = 8;    // u32 counts per scan thread
constexpr int SCAN_TILE = SCAN_THREADS * SCAN_ITEMS;

constexpr int64_t CHUNK_CHARS = 400000;  // safe chunking: window length, characters
constexpr int64_t RUN_CHARS = 25000;     // safe chunking: longest run, characters

constexpr uint32_t SPIN_LIMIT = 1u << 22;  // bounded waits (x ~100 ns each)

constexpr uint32_t PTOK_SPECIAL = 0x80000000u;
constexpr uint32_t PTOK_MASK = 0x7FFFFFFFu;

// Decoupled look-back descriptors: state in bits 63..62, value in 61..0.
constexpr uint64_t DESC_AGG = 1ull << 62;
constexpr uint64_t DESC_PREFIX = 2ull << 62;
constexpr uint64_t DESC_VAL = (1ull << 62) - 1;

// Device status block of one encode/decode (zeroed at the start of each call).
struct Status {
  int32_t code;      // first error (TK_E_*), 0 = none
  int32_t err_kind;  // which wait timed out, for diagnostics
  int64_t err_pos;   // smallest invalid UTF-8 byte offset (INT64_MAX if none)
  int64_t n_ptok;    // pre-tokens found by the split
  int64_t n_ids;     // ids produced (may exceed the output capacity)
  uint32_t n_long;   // pre-tokens over SHORT_MAX bytes (the long-piece lists)
  uint32_t n_mid_a;  // mid pieces of MID_MIN..8 bytes (front of mid_list)
  uint32_t n_mid_b;  // mid pieces of 9..SHORT_MAX bytes (back of mid_list)
  uint32_t n_own_a;  // distinct mid pieces (first occurrences) of each list, in mid_own
  uint32_t n_own_b;
  uint32_t n_medium;    // work list sizes and cursors of k_merge_global
  uint32_t n_biglong;
  uint32_t medium_next;
  uint32_t big_next;
  uint32_t big_next2;
  uint32_t dedup_big_next;
  uint32_t n_huge;       // entries of huge_list
  uint32_t n_cl;         // entries of cl_list
  uint32_t cl_next;
  int32_t holdback;      // streaming decode: bytes held back at the end
  uint32_t tail;         // ... and those bytes, little-endian
  uint32_t n_cache_hits;     // long pieces found in the cross-call cache
  uint32_t n_cache_inserts;  // long pieces added to it
  uint32_t tile_ctr[8];  // dynamic tile counters of the persistent kernels
  int64_t n_tiles;       // split tiles of this call (element count of the tile scan)
};

// Lookup tables of a tokenizer, in device memory (passed by value).
struct Tables {
  const uint32_t* byte_id;     // [256] id of each single byte
  const uint32_t* dense;       // [65536] rank of the two-byte token (a<<8|b), or RANK_MAX
  const uint64_t* pair_slots;  // open addressing: (a << 40) | (b << 20) | rank; empty = ~0
  uint32_t pair_log2;          // log2(number of slots)
  uint32_t pair_max_probe;     // longest probe sequence present in the table
  const uint8_t* ext_low;      // [max_id + 1] bit 0: a token a||x ranks below x; bit 1:
                               // a token x||b does (x = the id; a, b tokens)
  const uint64_t* s34_slots;   // open addressing over the 3- and 4-byte tokens:
                               // (bytes << 21) | (len == 4) << 20 | rank; empty = ~0
  uint32_t s34_log2;
  uint32_t s34_max_probe;
  const uint8_t* spec_bytes;   // specials, concatenated
  const int32_t* spec_off;     // [n_spec + 1]
  const int32_t* spec_ids;     // [n_spec]
  int32_t n_spec;
  uint32_t spec_first[8];      // 256-bit mask of the specials' first bytes
  const uint32_t* tok_start;   // [max_id + 1] decode: byte offset in tok_bytes
  const int32_t* tok_len;      // [max_id + 1] decode: length, -1 if the id is unused
  const uint8_t* tok_bytes;
  int64_t max_id;
  int32_t pattern;             // TK_PATTERN_CL100K or TK_PATTERN_R50K_DIGITS
};

// Cross-call word cache: merged ids of pre-tokens over SHORT_MAX bytes, kept
// between calls.  An entry holds the piece's bytes and ids; a slot maps the
// dedup key of the bytes to entry index + 1 (key 0 = empty slot).
struct CacheEntry {
  uint64_t byte_off, id_off;
  uint32_t len, n_ids;
};
struct CacheDev {
  unsigned long long* slots;  // [2 << slot_log2]: key, entry + 1
  CacheEntry* entries;
  uint8_t* bytes;
  int32_t* ids;
  unsigned long long* used;   // [3]: entries, bytes, ids reserved so far
  uint32_t slot_log2;
  uint64_t max_entries, max_bytes, max_ids;
};
constexpr uint32_t GSRC_CACHED = 0x80000000u;  // gsrc flag: an owner whose ids came from the cache

// Device scratch of one encode (all sized from max_bytes / max_segments).
struct Work {
  Status* status;
  uint64_t* desc_a;     // split: N-run carry chain, one per split tile
  uint64_t* desc_b;     // split: pre-token count chain
  uint64_t* desc_c;     // count scan chain
  uint64_t* desc_w;     // safe chunking: window scan chain
  uint64_t* desc_r;     // safe chunking: run scan chain
  uint32_t* win_cut;    // bitmap: 400k-character window cuts
  uint32_t* run_cut;    // bitmap: 25k-character run cuts
  uint32_t* pbits;      // bitmap: pre-token starts (written by the split)
  uint32_t* sbits;      // bitmap: special-token starts
  uint32_t* tile_first; // per split tile: first pre-token start (tile-relative) or ~0
  uint32_t* cnt;        // [max_bytes + 1] decode: bytes per id
  uint32_t* offs;       // [max_bytes + 1] decode: exclusive scan of cnt
  int32_t* arena;       // [max_bytes] ids of pieces merged through global memory, at their byte offset
  uint32_t* long_list;  // (start, length) of pre-tokens of SHORT_MAX+1 .. MEDIUM_MAX bytes
  uint32_t* mid_list;   // (start, length) of pre-tokens of MID_MIN .. SHORT_MAX bytes:
                        // up to 8 bytes from the front, longer ones from the back
  int64_t mid_cap;      // entries of mid_list (and of mid_own)
  uint32_t* mid_own;    // the distinct mid pieces, laid out as mid_list
  unsigned long long* mtab;  // dedup table of mid pieces: 4 words per slot (key, key2, owner | len, -)
  uint32_t mtab_log2;        // slots of this call: 2^mtab_log2 (cleared by k_clear_mtab)
  int mid_side;              // mid pieces are merged on a side stream (large calls), else in the tile kernel
  int mid_dedup;             // this call uses the mid-piece word cache (large calls)
  uint32_t mtab_log2_max;
  uint32_t* big_list;   // (start, length) of pre-tokens of MEDIUM_MAX+1 .. CLUSTER_MIN bytes
  uint32_t* cl_list;    // (start, length) of pre-tokens longer than CLUSTER_MIN bytes
  uint32_t* staging;    // per split tile: compacted short ids, long-piece table at the end
  uint32_t* tile_count; // per split tile: ids (then: exclusive scan -> tile_base)
  uint32_t* tile_base;  // [n_tiles + 1]
  uint32_t* tile_meta;  // per split tile: short ids (low 16 bits) | pieces merged outside << 16
  uint32_t* seg_rel;    // [max_segments + 1] ids before each segment start, within its tile
  uint32_t* tile_segs;  // per split tile: first segment index at or after t0 - HALO, t0,
                        // t0 + TILE, t0 + TILE + HALO
  uint32_t* gsrc;       // [max_bytes] at each long piece's start: the start of the identical
                        // piece whose merge it uses (itself for the first occurrence)
  unsigned long long* dtab;  // dedup table of long pieces: pairs (hash key, owner+1 | len << 32)
  uint32_t dtab_log2;
  uint32_t* lrk;        // [max_bytes] long merge: pair ranks
  uint32_t* lids2;      // [max_bytes] long merge: second id buffer
  uint32_t* lrk2;       // [max_bytes] long merge: second rank buffer
  uint8_t* lsel;        // [max_bytes] long merge: selection flags
  uint8_t* lchg;        // [max_bytes] long merge: changed flags
  uint64_t* huge_list;  // (output position, arena start, id count) of the long pieces
                        // whose ids the whole grid copies
  uint64_t* long_key;   // dedup key of each long_list / big_list / cl_list entry
  uint64_t* big_key;
  uint64_t* cl_key;
  CacheDev cache;       // the attached cross-call cache (use_cache) ...
  int use_cache;
  int64_t max_bytes;
  int64_t max_segments;
};

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// A self-contained descriptor (state and value in one 64-bit word) needs no
// ordering with other data: a relaxed store publishes it without the fence a
// release store implies.
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void set_error(Status* st, int code, int kind) {
  if (atomicCAS(&st->code, 0, code) == 0) st->err_kind = kind;
}

struct SumOp {
  __device__ static uint64_t id() { return 0; }
  __device__ static uint64_t comb(uint64_t l, uint64_t r) { return l + r; }
};
// Decoupled look-back, run by all 32 lanes of one warp: publishes the tile's
// aggregate, inspects 32 predecessors per step (ballots for their states, an
// ordered shuffle reduction for their values) until it meets an inclusive
// prefix, publishes its own inclusive prefix and returns the exclusive one on
// every lane.  Waits are bounded (TK_E_TIMEOUT).
template <class Op>
__device__ uint64_t chain_exclusive_warp(uint64_t* desc, int64_t tile, uint64_t agg, Status* st,
                                         int kind) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
    if (lane == 0) st_release_u64(&desc[0], DESC_PREFIX | agg);
    return Op::id();
  }
  if (lane == 0) st_release_u64(&desc[tile], DESC_AGG | agg);
  uint64_t acc = Op::id();
  int64_t j = tile - 1;
  uint32_t spins = 0;
  for (;;) {
    const int64_t idx = j - lane;  // lane 0 = nearest predecessor
    const uint64_t d = (idx >= 0) ? ld_acquire_u64(&desc[idx]) : (DESC_PREFIX | Op::id());
    const uint64_t state = d & ~DESC_VAL;
    const uint32_t pmask = __ballot_sync(0xffffffffu, state == DESC_PREFIX);
    const uint32_t rmask = __ballot_sync(0xffffffffu, state != 0);
    const int fp = pmask ? __ffs(pmask) - 1 : 31;
    const uint32_t need = (fp == 31) ? 0xffffffffu : ((2u << fp) - 1u);
    if ((rmask & need) != need) {
      if (++spins > SPIN_LIMIT) {
        if (lane == 0) set_error(st, TK_E_TIMEOUT, kind);
        break;
      }
      __nanosleep(32);
      continue;
    }
    // combine lanes fp..0 in tile order (a higher lane is an earlier tile)
    uint64_t x = (lane <= fp) ? (d & DESC_VAL) : Op::id();
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x = Op::comb(y, x);
    }
    acc = Op::comb(__shfl_sync(0xffffffffu, x, 0), acc);
    if (pmask) break;
    j -= 32;
  }
  if (lane == 0) st_release_u64(&desc[tile], DESC_PREFIX | Op::comb(acc, agg));
  return acc;
}

// The tables the merge loop reads, passed by value into the hot loops.
struct MergeTabs {
  const uint32_t* byte_id;
  const uint32_t* dense;
  const uint64_t* pair_slots;
  uint32_t pair_log2;
  uint32_t pair_max_probe;
  const uint64_t* s34_slots;
  uint32_t s34_log2;
  uint32_t s34_max_probe;
  __device__ __host__ explicit MergeTabs(const Tables& T)
      : byte_id(T.byte_id), dense(T.dense), pair_slots(T.pair_slots), pair_log2(T.pair_log2),
        pair_max_probe(T.pair_max_probe), s34_slots(T.s34_slots), s34_log2(T.s34_log2),
        s34_max_probe(T.s34_max_probe) {}
};

// Slot of a 3- or 4-byte slice (bytes little-endian in a 32-bit key) in the
// slice table.
__host__ __device__ __forceinline__ uint32_t s34_hash(uint32_t key, uint32_t log2) {
  return (key * 0x9E3779B1u) >> (32 - log2);
}

// Load that bypasses L1 allocation (the streamed text), keeping L1 for the
// small tables the merge reads on every pre-token.
__device__ __forceinline__ uint4 ld_na_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Rank of the two-byte token b0 b1, or RANK_MAX (the dense first-round table;
// one L2-resident load measured faster than any compressed form).
__device__ __forceinline__ uint32_t dense_rank(const MergeTabs& T, uint32_t b0, uint32_t b1) {
  return __ldg(&T.dense[(b0 << 8) | b1]);
}

// Carry of an operator whose aggregate can "reset" (the number-run and the
// segmented code-point counts): every tile publishes its aggregate first
// (st_release of DESC_AGG | agg); this walk then combines
// the predecessors' aggregates backwards only until one that resets (the
// carry cannot depend on anything before it).  No inclusive prefixes are
// published or awaited, so a tile waits only for the few predecessors its
// carry really depends on, each of which publishes early.  Run by one warp;
// `resets(v)` tells whether aggregate v resets.  Bounded waits.
template <class Op>
__device__ uint64_t carry_walk_warp(uint64_t* desc, int64_t tile, uint64_t agg, Status* st, int kind) {
  const int lane = threadIdx.x & 31;
  (void)agg;
  uint64_t acc = Op::id();
  int64_t j = tile - 1;
  uint32_t spins = 0;
  while (j >= 0) {
    const int64_t idx = j - lane;
    const uint64_t d = (idx >= 0) ? ld_acquire_u64(&desc[idx]) : (DESC_AGG | Op::reset_id());
    const bool ready = (d & ~DESC_VAL) != 0;
    const uint64_t v = d & DESC_VAL;
    const uint32_t rst = __ballot_sync(0xffffffffu, ready && Op::resets(v));
    const uint32_t rdy = __ballot_sync(0xffffffffu, ready);
    const int fr = rst ? __ffs(rst) - 1 : 31;
    const uint32_t need = (fr == 31) ? 0xffffffffu : ((2u << fr) - 1u);
    if ((rdy & need) != need) {
      if (++spins > SPIN_LIMIT) {
        if (lane == 0) set_error(st, TK_E_TIMEOUT, kind);
        break;
      }
      __nanosleep(32);
      continue;
    }
    uint64_t x = (lane <= fr) ? v : Op::id();
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x = Op::comb(y, x);
    }
    acc = Op::comb(__shfl_sync(0xffffffffu, x, 0), acc);
    if (rst) break;
    j -= 32;
  }
  return acc;
}

// Open-addressing lookup of the rank of the token whose bytes are
// bytes(a) || bytes(b), or RANK_MAX.
template <class TT>
__device__ __forceinline__ uint32_t pair_rank(const TT& T, uint32_t a, uint32_t b) {
  const uint64_t key = ((uint64_t)a << 20) | b;
  uint64_t h = (key * 0x9E3779B97F4A7C15ull) >> (64 - T.pair_log2);
  const uint64_t mask = (1ull << T.pair_log2) - 1;
  for (uint32_t probe = 0; probe <= T.pair_max_probe; probe++) {
    const uint64_t s = __ldg(&T.pair_slots[h]);
    if (s == ~0ull) return RANK_MAX;
    if ((s >> 20) == key) return (uint32_t)(s & 0xFFFFF);
    h = (h + 1) & mask;
  }
  return RANK_MAX;
}

// The same lookup in two steps, so that a thread can have several first
// probes in flight: pair_first loads the first slot (none when `use` is
// false), pair_finish resolves it, probing on past a collision.
struct PairProbe {
  uint64_t s, key;
};
template <class TT>
__device__ __forceinline__ PairProbe pair_first(const TT& T, uint32_t a, uint32_t b, bool use) {
  PairProbe p;
  p.key = ((uint64_t)a << 20) | b;
  p.s = use ? __ldg(&T.pair_slots[(p.key * 0x9E3779B97F4A7C15ull) >> (64 - T.pair_log2)]) : ~0ull;
  return p;
}
template <class TT>
__device__ __forceinline__ uint32_t pair_finish(const TT& T, PairProbe p) {
  if (p.s == ~0ull) return RANK_MAX;
  if ((p.s >> 20) == p.key) return (uint32_t)(p.s & 0xFFFFF);
  const uint64_t mask = (1ull << T.pair_log2) - 1;
  uint64_t h = (p.key * 0x9E3779B97F4A7C15ull) >> (64 - T.pair_log2);
  for (uint32_t probe = 1; probe <= T.pair_max_probe; probe++) {
    h = (h + 1) & mask;
    const uint64_t s = __ldg(&T.pair_slots[h]);
    if (s == ~0ull) return RANK_MAX;
    if ((s >> 20) == p.key) return (uint32_t)(s & 0xFFFFF);
  }
  return RANK_MAX;
}

// Rank of the 3- or 4-byte slice `key` (RANK_MAX if it is not a token),
// given the slot `s` its first probe read (loaded early, so that this load
// overlaps the pair loads it does not depend on).
template <class TT>
__device__ __forceinline__ uint32_t s34_rank(const TT& T, uint64_t s, uint32_t key, bool four) {
  const uint64_t k = ((uint64_t)key << 1) | (four ? 1u : 0u);
  uint32_t h = s34_hash(key, T.s34_log2);
  for (uint32_t probe = 0;;) {
    if (s == ~0ull) return RANK_MAX;
    if ((s >> 20) == k) return (uint32_t)(s & 0xFFFFF);
    if (++probe > T.s34_max_probe) return RANK_MAX;
    h = (h + 1) & ((1u << T.s34_log2) - 1u);
    s = __ldg(&T.s34_slots[h]);
  }
}

template <class TT>
__device__ __forceinline__ uint64_t s34_first(const TT& T, uint32_t key) {
  return __ldg(&T.s34_slots[s34_hash(key, T.s34_log2)]);
}

}  // namespace tk

struct tk_tokenizer {
  tk::Tables t;
  static constexpr int MAX_DEV = 32;
  void* dev_mem[MAX_DEV];
  int n_dev;
  int64_t n_ranks;
  int device;
  int num_sms;
};

struct tk_profile {
  static constexpr int MAXK = 64;
  int on;
  int n;                        // kernels with totals
  const char* names[MAXK];
  double total_ms[MAXK];
  int64_t launches[MAXK];
  cudaEvent_t ev[MAXK + 1];     // events of the call in flight, one per mark
  const char* pending[MAXK];    // kernel starting at each mark (null: an end mark)
  cudaStream_t pstream[MAXK];   // the stream of each mark
  int n_pending;
};

struct tk_cache {
  tk::CacheDev d;
  const tk_tokenizer* tok;
  static constexpr int MAX_DEV = 8;
  void* dev_mem[MAX_DEV];
  int n_dev;
  int device;
};

struct tk_workspace {
  tk::Work w;
  tk_profile prof;
  const tk_tokenizer* tok;
  tk_cache* cache;  // attached cross-call cache, or null
  static constexpr int MAX_DEV = 64;
  void* dev_mem[MAX_DEV];
  int n_dev;
  tk::Status* h_status;     // pinned host copy of the status block
  int split_per_sm, scan_per_sm, copy_per_sm;  // resident CTAs per SM (0: not queried yet)
  uint8_t* d_stage_text;    // staging for tk_encode_segments_host
  int64_t* d_stage_off;
  uint8_t* d_stage_allow;
  int32_t* d_stage_ids;
  int64_t* d_stage_offsets;
  // pipelined host calls: the text is cut at segment boundaries into batches
  // whose copies in and out overlap the encode of their neighbours
  static constexpr int PIPE_MAX = 16;
  cudaStream_t s_h2d, s_d2h;
  cudaStream_t s_side;               // the long-piece kernels, next to the tile kernel
  cudaStream_t s_mid;                // the mid-piece kernels, next to both
  cudaStream_t s_cl, s_med;          // the cluster and medium merges, next to the big merges
  cudaEvent_t ev_dedup, ev_cl, ev_med;  // fork after the long pieces' word cache, joins
  cudaEvent_t ev_split, ev_long;     // fork after the split, join before the fixup
  cudaEvent_t ev_find, ev_mid;       // fork after the listing, join before the fixup
  cudaEvent_t ev_start, ev_h2d[PIPE_MAX], ev_done[PIPE_MAX];
  int n_events;
  // a repeated device call (same tokenizer, buffers, sizes and cache) is
  // captured into a graph the second time it comes and replayed after that,
  // on s_graph, joined with the caller's stream by events
  cudaStream_t s_graph;
  cudaEvent_t ev_gin, ev_gout;
  cudaGraphExec_t g_exec;
  uint64_t g_key[12];
  int g_seen;  // calls in a row with g_key
  int g_off;   // a capture failed: no graphs for this workspace
  int prio_hi; // the side streams' priority (the graph's side kernels get it too)
  tk::Status* h_pipe_status;  // [PIPE_MAX] pinned
  int64_t* d_stage_raw;       // segment offsets as copied in, before rebasing
  int64_t* d_pipe_base;       // [PIPE_MAX + 1] ids before each batch
  int device;
  int num_sms;
};

// Internal C++ entry points shared between translation units.
void tk_set_error(const char* fmt, ...);
// Profiling helpers: mark() before a launch (records an event when profiling
// is on); finish() after the call's synchronisation adds up the durations.
// Marks the start of `kernel` on stream st (kernel null: the end of the previous
// kernel on st).  A kernel's time runs from its mark to the next mark on the
// same stream, so kernels on several streams keep running concurrently.
void tk_prof_mark(tk_workspace* ws, const char* kernel, cudaStream_t st);
void tk_prof_finish(tk_workspace* ws, cudaStream_t st);
int tk_scan_u32(tk_workspace* ws, const uint32_t* d_in, uint32_t* d_out, const int64_t* d_n,
                int64_t n_max, int chain_ctr, cudaStream_t st);
